"""The allocation-free scoring call (spinf_score_static) against the regular one.

Some callers cannot allocate device memory while they serve (a memory budget
fixed at start-up, an allocator they do not control); spinf_score_static keeps
its scratch in the library's own fixed device array instead of a caller
workspace.  It runs the same kernels, in the same fixed reduction order, on the
same inputs as spinf_score, so its results must be bit-identical to spinf_score's,
call after call: any difference would be stale scratch left in the shared array
by an earlier call.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_score
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _static(spinf, plan, p, h, w, w_scale, w_dtype, shape):
    info = plan.pass_info(p)
    lse = torch.full((info.M,), float("nan"), device="cuda")
    tlp = torch.full((info.G,), float("nan"), device="cuda")
    spinf.score_static(plan, p, h, w, w_scale, w_dtype, shape.d_model, shape.vocab, lse, tlp)
    plan.device_status()
    torch.cuda.synchronize()
    return lse.cpu().numpy(), tlp.cpu().numpy()


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
def test_static_scratch_matches_workspace_call(spinf, fp8):
    # two different passes in a row, then the first again: the shared array is reused
    shape = wl.Shape(4, 2, 64, 512, 1000)
    inputs = wl.stress(n_questions=80, content_tokens=100, vocab=1000)
    P = oracle_plan(inputs, vocab=1000)
    plan = spinf.Plan(inputs, vocab=1000)
    w = sv.lm_head(shape.vocab, shape.d_model)
    w_dtype = spinf.DTYPE_E4M3 if fp8 else spinf.DTYPE_BF16
    w_scale = None
    if fp8:
        w, w_scale = sv.e4m3_rows(w)
        w_scale = w_scale.cuda()
    w = w.cuda()
    hs = []
    for p, lay in enumerate(P.passes):
        _, _, _, h = pass_values(lay, shape)
        hs.append(h)
    order = [0, len(P.passes) - 1, 0]
    for p in order:
        ref_lse, ref_tlp, _ = run_score(spinf, plan, p, hs[p], w, w_scale, w_dtype, shape)
        for _ in range(2):
            lse, tlp = _static(spinf, plan, p, hs[p], w, w_scale, w_dtype, shape)
            assert np.array_equal(lse, ref_lse)   # bitwise: same kernels, same order, same inputs
            assert np.array_equal(tlp, ref_tlp)


def test_static_scratch_rejects_oversized_pass(spinf):
    inputs = wl.tiny()
    plan = spinf.Plan(inputs, vocab=1024)
    plan.upload(0)
    d_model = 1 << 20            # 128 rows x 2^20 bf16 = 256 MiB of gathered rows: beyond the area
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    a = x.data_ptr()   # raw addresses: the library's own limit check runs, not the binding's size checks
    with pytest.raises(spinf.SpinfError) as e:
        spinf.score_static(plan, 0, a, a, None, spinf.DTYPE_BF16, d_model, 1024, a, a)
    assert e.value.status_name == "LIMIT"
    assert "static area holds" in str(e.value)
