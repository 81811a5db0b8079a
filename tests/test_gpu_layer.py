"""GPU steps around the attention call against the layer oracle: rotary positions at
tree depth (spinf_rope_tree), the projections on the tensor cores (spinf_linear,
spinf_qkv_rope with the rotary turn fused), their e4m3 form with static scales, and
the packed layer."""
import math

import numpy as np
import pytest
import torch

from gpu_util import oracle_plan, pass_values, run_attention
from oracle import layer as ol
from synth import values as sv
from synth import workloads as wl

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rope_tree_matches_oracle(spinf, d):
    inputs = wl.stress(n_questions=24, content_tokens=300, vocab=1000) + wl.tiny(vocab=1000)
    lay = oracle_plan(inputs, token_budget=1024, vocab=1000).passes[0]
    plan = spinf.Plan(inputs, token_budget=1024, vocab=1000)
    plan.upload(0)
    q, k, _, _ = pass_values(lay, wl.Shape(8, 2, d, 256, 1000), hidden_rows=False)
    ref_q = ol.rope(q.float().cpu().numpy(), lay.pos, 10000.0)
    ref_k = ol.rope(k.float().cpu().numpy(), lay.pos, 10000.0)
    spinf.rope_tree(plan, 0, q, k, 8, 2, d, 10000.0)
    plan.device_status()
    for got, ref in ((q, ref_q), (k, ref_k)):
        got = got.float().cpu().numpy()
        assert np.all(np.abs(got - ref) <= 2 ** -7 * np.abs(ref) + 1e-3)


def test_rope_tree_is_packing_invariant(spinf):
    target = wl.stress(n_questions=12, content_tokens=230, vocab=1000)[0]
    others = wl.short_inputs(vocab=1000, n=40)
    outs = []
    for offset in (0, 5, 21):
        inputs = others[:offset] + [target] + others[offset:]
        lay = oracle_plan(inputs, vocab=1000, floors=False).passes[0]
        plan = spinf.Plan(inputs, vocab=1000, floors=False)
        plan.upload(0)
        q, k, _, _ = pass_values(lay, wl.Shape(8, 2, 128, 256, 1000), hidden_rows=False)
        spinf.rope_tree(plan, 0, q, k, 8, 2, 128, 10000.0)
        u = next(u for u in lay.units if u.source == offset)
        outs.append((q[u.start:u.start + u.size].clone(), k[u.start:u.start + u.size].clone()))
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1])


def _tiny_plan(spinf):
    inputs = wl.tiny()
    plan = spinf.Plan(inputs, vocab=1024)
    plan.upload(0)
    return plan


def _within_bf16(got, ref, ulps=2.0, atol=1e-3):
    """|got - ref| within `ulps` bf16 ulps of |ref| (2^-8 relative each) plus atol."""
    return np.all(np.abs(got - ref) <= ulps * 2 ** -8 * np.abs(ref) + atol)


@pytest.mark.parametrize("rows,K,N", [(300, 256, 512), (128, 3840, 768), (77, 520, 96)])
def test_linear_bf16_matches_oracle(spinf, rows, K, N):
    """Ragged rows and features (several tiles, a partial last tile in both directions)."""
    plan = _tiny_plan(spinf)
    g = np.random.default_rng(rows)
    x = _bf16(g.normal(size=(rows, K))).cuda()
    w = _bf16(g.normal(size=(N, K)) / math.sqrt(K)).cuda()
    y = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    spinf.linear(plan, x, w, y)
    plan.device_status()
    ref = x.double().cpu().numpy() @ w.double().cpu().numpy().T
    assert _within_bf16(y.float().cpu().numpy(), ref)


def test_linear_rows_do_not_depend_on_the_batch(spinf):
    plan = _tiny_plan(spinf)
    g = np.random.default_rng(9)
    x = _bf16(g.normal(size=(600, 512))).cuda()
    w = _bf16(g.normal(size=(1024, 512)) / 16).cuda()
    full = torch.empty(600, 1024, dtype=torch.bfloat16, device="cuda")
    spinf.linear(plan, x, w, full)
    for a, b in ((37, 150), (0, 1), (129, 600)):
        part = torch.empty(b - a, 1024, dtype=torch.bfloat16, device="cuda")
        spinf.linear(plan, x[a:b], w, part)
        plan.device_status()
        assert torch.equal(part, full[a:b])


def test_linear_e4m3_static_scales(spinf):
    """Codes of the activations bit for bit against the oracle; the product within the
    fp8 tolerance of the oracle's fp64 product of the same codes and scales."""
    plan = _tiny_plan(spinf)
    g = np.random.default_rng(11)
    rows, K, N = 260, 1024, 512
    x = _bf16(g.normal(size=(rows, K))).cuda()
    w = _bf16(g.normal(size=(N, K)) / 32)
    w_codes, w_scale = sv.e4m3_rows(w)
    x_scale = np.float32(4.5 / 448)   # a static scale (a calibration stand-in)
    codes = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    spinf.quantize_static(x, float(x_scale), codes)
    torch.cuda.synchronize()
    want = ol.quantize_static(x.float().cpu().numpy(), x_scale)
    np.testing.assert_array_equal(codes.cpu().numpy(), want)
    y = torch.empty(rows, N, dtype=torch.bfloat16, device="cuda")
    spinf.linear(plan, codes, w_codes.cuda(), y, w_scale=w_scale.cuda(), x_scale=float(x_scale),
                 w_dtype=spinf.DTYPE_E4M3)
    plan.device_status()
    ref = ol.linear_fp8(want, x_scale, w_codes.numpy(), w_scale.numpy())
    assert _within_bf16(y.float().cpu().numpy(), ref)


def _qkv_case(spinf, shape, inputs, dtype):
    Hq, Hkv, d, D = shape.n_q_heads, shape.n_kv_heads, shape.d_head, shape.d_model
    lay = oracle_plan(inputs, vocab=shape.vocab).passes[0]
    plan = spinf.Plan(inputs, vocab=shape.vocab)
    plan.upload(0)
    keys = sv.path_keys(lay.tok, lay.parent, lay.T)
    x = sv.hidden(keys, lay.T_pad, D).cuda()
    g = np.random.default_rng(d)
    w = _bf16(g.normal(size=((Hq + 2 * Hkv) * d, D)) / math.sqrt(D))
    q = torch.full((lay.T_pad, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    k = torch.full((lay.T_pad, Hkv, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    v = torch.full_like(k, float("nan"))
    if dtype == "bf16":
        spinf.qkv_rope(plan, 0, x, w.cuda(), q, k, v, Hq, Hkv, d)
        xr, wr = x.float().cpu().numpy(), w.float().numpy()
    else:
        x_scale = np.float32(5.0 / 448)
        codes = torch.empty(lay.T_pad, D, dtype=torch.uint8, device="cuda")
        spinf.quantize_static(x, float(x_scale), codes)
        w_codes, w_scale = sv.e4m3_rows(w)
        spinf.qkv_rope(plan, 0, codes, w_codes.cuda(), q, k, v, Hq, Hkv, d, w_scale=w_scale.cuda(),
                       x_scale=float(x_scale), w_dtype=spinf.DTYPE_E4M3)
        from oracle import fp8
        xr = fp8.decode(ol.quantize_static(x.float().cpu().numpy(), x_scale)) * float(x_scale)
        wr = fp8.decode(w_codes.numpy()) * w_scale.numpy().astype(np.float64)[:, None]
    plan.device_status()
    rq, rk, rv = ol.qkv_rope(xr, wr, lay.pos, Hq, Hkv, d, 10000.0)
    T = lay.T
    for got, ref in ((q, rq), (k, rk), (v, rv)):
        assert _within_bf16(got[:T].float().cpu().numpy(), ref[:T])
    return lay, plan, (q, k, v), (xr, wr)


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("shape_name", ["tiny", "qwen", "gemma"])
def test_qkv_rope_matches_oracle(spinf, dtype, shape_name):
    """Fused projection + rotary at tree depth: q, k, v against the oracle, d_head 64 / 128 / 256
    (the tiny shape's k and v heads end inside a 256-column tile)."""
    if shape_name == "tiny":
        shape, inputs = wl.TINY, wl.tiny()
    elif shape_name == "qwen":
        shape, inputs = wl.Shape(40, 8, 128, 1024, 1000), wl.stress(n_questions=12, content_tokens=200, vocab=1000)
    else:
        shape, inputs = wl.Shape(16, 8, 256, 768, 1000), wl.stress(n_questions=12, content_tokens=200, vocab=1000)
    _qkv_case(spinf, shape, inputs, dtype)


def test_qkv_rope_is_packing_invariant(spinf):
    shape = wl.Shape(8, 2, 128, 512, 1000)
    target = wl.stress(n_questions=10, content_tokens=150, vocab=1000)[0]
    others = wl.short_inputs(vocab=1000, n=40)
    g = np.random.default_rng(3)
    w = _bf16(g.normal(size=(12 * 128, 512)) / 24).cuda()
    outs = []
    for offset in (0, 7, 40):
        inputs = others[:offset] + [target] + others[offset:]
        lay = oracle_plan(inputs, vocab=1000, floors=False).passes[0]
        plan = spinf.Plan(inputs, vocab=1000, floors=False)
        plan.upload(0)
        keys = sv.path_keys(lay.tok, lay.parent, lay.T)
        x = sv.hidden(keys, lay.T_pad, 512).cuda()
        q = torch.empty(lay.T_pad, 8, 128, dtype=torch.bfloat16, device="cuda")
        k = torch.empty(lay.T_pad, 2, 128, dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        spinf.qkv_rope(plan, 0, x, w, q, k, v, 8, 2, 128)
        plan.device_status()
        u = next(u for u in lay.units if u.source == offset)
        sl = slice(u.start, u.start + u.size)
        outs.append((q[sl].clone(), k[sl].clone(), v[sl].clone()))
    for got in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(got, outs[0]))


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_packed_layer_matches_oracle(spinf, dtype):
    """x -> fused QKV + rotary at tree depth -> attention -> output projection on a packed pass."""
    shape = wl.TINY
    Hq, Hkv, d, D = shape.n_q_heads, shape.n_kv_heads, shape.d_head, shape.d_model
    inputs = wl.stress(n_questions=10, content_tokens=150, vocab=1024) + wl.tiny()
    lay, plan, (q, k, v), (xr, wr) = _qkv_case(spinf, shape, inputs, dtype)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    g = np.random.default_rng(5)
    w_o = _bf16(g.normal(size=(D, Hq * d)) / math.sqrt(Hq * d))
    out = torch.empty(lay.T_pad, D, dtype=torch.bfloat16, device="cuda")
    spinf.linear(plan, o.view(lay.T_pad, Hq * d), w_o.cuda(), out)
    plan.device_status()
    rows = list(range(lay.T))
    # the oracle takes the projection's inputs as the kernels saw them (bf16 values, or the
    # e4m3 codes times their static scales), in fp64
    ref = ol.packed_layer_rows(lay, xr, wr, w_o.float().numpy(), Hq, Hkv, d, 10000.0, rows)
    assert np.abs(out[:lay.T].float().cpu().numpy() - ref).max() <= 5e-2
