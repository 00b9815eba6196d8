"""The score-then-select scorer (DS4X_SCORER=two_stage: every row's key
written to the workspace, then a radix select of the top-k) against the
oracle.  The variable is read once per process, so the cases run in a child
process with it set."""

import os
import subprocess
import sys

import pytest

from gpu_path import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import numpy as np
from gpu_path import pack, score_topk
from oracle import codecs as C, indexer as I
from parity import check_topk
from synth import decode_case, to_bf16_bits
for n, k in [(1, 512), (513, 512), (4096, 512), (20000, 7), (131072, 512), (300000, 100)]:
    case = decode_case(n, 3000 + n) if n <= 20000 else None
    if case is None:
        from synth import indexer_case
        case = indexer_case(n, 3000 + n)
    rows, _ = pack(idx_in=case["idx_in"])
    gi, gs = score_topk(rows, n, case["q_idx"], case["w"], k)
    check_topk(gi, gs, I.score_rows(C.pack_idx_rows(case["idx_in"]), case["q_idx"], case["w"]), k)
# all-equal scores: the tie break by index
case = decode_case(5000, 11)
rows, _ = pack(idx_in=case["idx_in"])
gi, gs = score_topk(rows, 5000, np.zeros((64, 128), np.uint16), case["w"], 512)
assert np.array_equal(gi, np.arange(512)) and np.all(gs == 0)
print("two-stage ok")
"""


def test_two_stage_scorer_parity():
    require_gpu()
    env = dict(os.environ, DS4X_SCORER="two_stage")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "two-stage ok" in r.stdout
