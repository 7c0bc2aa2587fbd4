"""Merged chunk launches change no bit of any output.

Both fused steps run two chunks' projections as one GEMM launch: the step with
the backward recompute runs chunk c's G with chunk c+1's forward, the step
without it the forward GEMMs of chunks c and c+1 (c even).  Each output tile is
computed by the same arithmetic either way, so every output must equal, bit for
bit, what separate launches give (KD_MERGE_LOGITS=0, read once per process,
hence a child process).  Long-context head, 2048-row chunks: T 6444 is four
chunks with a ragged last one, T 5000 three chunks, the last one without a
partner in the step without the recompute."""
import os
import subprocess
import sys

import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_inputs
from parity_util import to_dev

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [(step, T) for step in ("fused_step", "fused_step_norecompute") for T in (6444, 5000)]
KEYS = ("loss", "lse", "loss_rows", "dH", "dW")

CHILD = """
import sys, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_inputs
from parity_util import to_dev
dev = torch.device('cuda:0')
out = {{}}
for step, T in {cases!r}:
    inp = make_inputs('longctx', device=dev, T=T)
    idx, p = to_dev(inp['idx'], inp['p'], dev)
    r = getattr(api, step)(inp['H'], inp['W'], idx, p, 2048, loss_rows=True)
    out[(step, T)] = {{k: r[k].cpu() for k in {keys!r}}}
torch.save(out, {dst!r})
"""


@pytest.fixture(scope="module")
def separate(tmp_path_factory):
    dst = str(tmp_path_factory.mktemp("merge") / "separate.pt")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), cases=CASES, keys=KEYS, dst=dst)
    env = dict(os.environ, KD_MERGE_LOGITS="0")
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-3000:]
    return torch.load(dst)


@pytest.mark.parametrize("step,T", CASES)
def test_merged_launches_match_separate_launches(cuda_device, separate, step, T):
    inp = make_inputs("longctx", device=cuda_device, T=T)
    idx, p = to_dev(inp["idx"], inp["p"], cuda_device)
    got = getattr(api, step)(inp["H"], inp["W"], idx, p, 2048, loss_rows=True)
    torch.cuda.synchronize()
    ref = separate[(step, T)]
    for k in KEYS:
        assert torch.equal(got[k].cpu(), ref[k]), k
