"""bench.py's roofline `traffic` figures are DRAM read + write bytes copied
from ncu summaries under profiles/: each must still name a summary that exists
and prints both of its byte counts, so that a re-capture that updates one side
and not the other shows up here."""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def traffic_constants():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    out = {}
    for node in tree.body:
        if not isinstance(node, ast.Assign) or len(node.targets) != 1:
            continue
        name = getattr(node.targets[0], "id", "")
        if not name.endswith("_TRAFFIC"):
            continue
        total, path = node.value.elts
        assert isinstance(total, ast.BinOp) and isinstance(total.op, ast.Add), name
        out[name] = (total.left.value, total.right.value, path.value)
    return out


def test_every_traffic_constant_matches_its_profile():
    consts = traffic_constants()
    assert set(consts) == {"DECODE_TRAFFIC", "PREFILL_TRAFFIC", "WRITE_TRAFFIC"}
    for name, (read, write, path) in consts.items():
        text = open(os.path.join(ROOT, path)).read()
        for label, value in (("dram__bytes_read.sum", read), ("dram__bytes_write.sum", write)):
            assert f"{label} {value:,} B" in text or f"| {label} | {value:,} B" in text, \
                (name, label, value, path)
