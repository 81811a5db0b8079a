"""End to end on the GPU: plan, attention, scoring and collect against the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_attention, run_score
from oracle import collect as oc
from oracle import score as osc
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def test_tiny_pipeline(spinf):
    inputs, shape = wl.tiny(), wl.TINY
    P = oracle_plan(inputs, vocab=shape.vocab)
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    w = sv.lm_head(shape.vocab, shape.d_model)
    gpu_lp, ref_lp = [], []
    for p, lay in enumerate(P.passes):
        q, k, v, h = pass_values(lay, shape)
        run_attention(spinf, plan, p, q, k, v, shape)
        _, tlp, _ = run_score(spinf, plan, p, h, w.cuda(), None, spinf.DTYPE_BF16, shape)
        gpu_lp.append(tlp)
        ref_lp.append(osc.score_rows(h.float().cpu().numpy()[lay.slot_row], lay.gather_m, lay.gather_tok,
                                     w=w.float().numpy())[1])
    ours = plan.collect(gpu_lp)
    ref = oc.collect(P, ref_lp)
    flat_lp = np.concatenate([r["lp"] for per_q in ref for r in per_q])
    flat_p = np.concatenate([r["p"] for per_q in ref for r in per_q])
    flat_fp = np.concatenate([r["floor_p"] for per_q in ref for r in per_q])
    res = np.array([r["residual"] for per_q in ref for r in per_q])
    assert np.abs(ours["option_lp"] - flat_lp).max() <= 4e-3
    assert np.abs(ours["option_p"] - flat_p).max() <= 4e-3
    assert np.abs(ours["option_floor_p"] - flat_fp).max() <= 4e-3
    assert np.abs(ours["residual"] - res).max() <= 4e-3


def test_upload_into_caller_memory_gives_identical_results(spinf):
    """spinf_plan_upload_to (descriptors and error word in caller-owned memory, reused by a
    second plan) against the plan-owned upload: bit-identical attention and scores."""
    inputs = wl.stress(n_questions=20, content_tokens=300, vocab=1024) + wl.tiny()
    shape = wl.TINY
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    q, k, v, h = pass_values(lay, shape)
    w = sv.lm_head(shape.vocab, shape.d_model).cuda()
    a = spinf.Plan(inputs, vocab=shape.vocab)
    o_a = run_attention(spinf, a, 0, q, k, v, shape)
    lse_a, tlp_a, _ = run_score(spinf, a, 0, h, w, None, spinf.DTYPE_BF16, shape)
    buf = torch.empty(a.descriptor_bytes(0) + 4096, dtype=torch.uint8, device="cuda")
    for _ in range(2):   # the same memory serves a second plan once the first is done
        b = spinf.Plan(inputs, vocab=shape.vocab)
        b.upload(0, buffer=buf)
        o_b = run_attention(spinf, b, 0, q, k, v, shape)
        lse_b, tlp_b, _ = run_score(spinf, b, 0, h, w, None, spinf.DTYPE_BF16, shape)
        assert torch.equal(o_a, o_b)
        assert np.array_equal(lse_a, lse_b) and np.array_equal(tlp_a, tlp_b)
        b.close()


def test_upload_from_pinned_staging_gives_identical_results(spinf):
    """spinf_plan_upload_pinned (descriptors written into caller-owned page-locked memory, then
    copied) against the plan-owned upload: bit-identical attention and scores; pageable or
    short staging is refused before any copy."""
    inputs = wl.stress(n_questions=20, content_tokens=300, vocab=1024) + wl.tiny()
    shape = wl.TINY
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    q, k, v, h = pass_values(lay, shape)
    w = sv.lm_head(shape.vocab, shape.d_model).cuda()
    a = spinf.Plan(inputs, vocab=shape.vocab)
    o_a = run_attention(spinf, a, 0, q, k, v, shape)
    lse_a, tlp_a, _ = run_score(spinf, a, 0, h, w, None, spinf.DTYPE_BF16, shape)
    need = a.descriptor_bytes(0)
    buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    b = spinf.Plan(inputs, vocab=shape.vocab)
    for bad in (torch.empty(need, dtype=torch.uint8),                       # pageable
                torch.empty(need - 257, dtype=torch.uint8).pin_memory()):  # short
        with pytest.raises(spinf.SpinfError) as e:
            b.upload(0, buffer=buf, staging=bad)
        assert e.value.status_name == "INVALID"
    stage = torch.full((need,), 0xAB, dtype=torch.uint8).pin_memory()   # stale bytes must not leak in
    b.upload(0, buffer=buf, staging=stage)
    o_b = run_attention(spinf, b, 0, q, k, v, shape)
    lse_b, tlp_b, _ = run_score(spinf, b, 0, h, w, None, spinf.DTYPE_BF16, shape)
    assert torch.equal(o_a, o_b)
    assert np.array_equal(lse_a, lse_b) and np.array_equal(tlp_a, tlp_b)
    b.close()


def test_bounded_wait_runs_out_and_device_stays_usable(spinf):
    """A device wait that nothing satisfies ends after its bound, the error word reports a
    timeout once, and the next calls on the same context run normally."""
    inputs, shape = wl.tiny(), wl.TINY
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    plan.upload(0)
    plan.device_selftest(wait_ms=30)
    with pytest.raises(spinf.SpinfError) as e:
        plan.device_status()
    assert e.value.status_name == "DEVICE_TIMEOUT"
    plan.device_status()   # cleared
    q, k, v, _ = pass_values(lay, shape, hidden_rows=False)
    o1 = run_attention(spinf, plan, 0, q, k, v, shape)
    o2 = run_attention(spinf, plan, 0, q, k, v, shape)
    assert torch.equal(o1, o2) and torch.isfinite(o1).all()


def test_selftest_rejects_bad_arguments(spinf):
    plan = spinf.Plan(wl.tiny(), vocab=1024)
    with pytest.raises(spinf.SpinfError):
        plan.device_selftest(30)          # nothing uploaded yet: no error word
    plan.upload(0)
    for bad in (0, 10001):
        with pytest.raises(spinf.SpinfError):
            plan.device_selftest(bad)
