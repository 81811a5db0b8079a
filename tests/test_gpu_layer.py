"""GPU steps around the attention call against the layer oracle: rotary positions at
tree depth (spinf_rope_tree), the projections (spinf_linear), the packed layer."""
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


def test_linear_matches_oracle(spinf):
    g = np.random.default_rng(4)
    x = _bf16(g.normal(size=(300, 256))).cuda()
    w = _bf16(g.normal(size=(512, 256)) / 16).cuda()
    y = torch.empty(300, 512, dtype=torch.bfloat16, device="cuda")
    spinf.linear(x, w, y)
    torch.cuda.synchronize()
    ref = x.double().cpu().numpy() @ w.double().cpu().numpy().T
    assert np.all(np.abs(y.float().cpu().numpy() - ref) <= 2 ** -8 * np.abs(ref) + 1e-3)


def test_packed_layer_matches_oracle(spinf):
    """x -> QKV -> rotary at tree depth -> attention -> output projection on a packed pass."""
    shape = wl.TINY
    Hq, Hkv, d, D = shape.n_q_heads, shape.n_kv_heads, shape.d_head, shape.d_model
    inputs = wl.stress(n_questions=10, content_tokens=150, vocab=1024) + wl.tiny()
    lay = oracle_plan(inputs, vocab=1024).passes[0]
    plan = spinf.Plan(inputs, vocab=1024)
    plan.upload(0)
    keys = sv.path_keys(lay.tok, lay.parent, lay.T)
    x = sv.hidden(keys, lay.T_pad, D).cuda()
    g = np.random.default_rng(5)
    w_qkv = _bf16(g.normal(size=((Hq + 2 * Hkv) * d, D)) / math.sqrt(D)).cuda()
    w_o = _bf16(g.normal(size=(D, Hq * d)) / math.sqrt(Hq * d)).cuda()
    y = torch.empty(lay.T_pad, (Hq + 2 * Hkv) * d, dtype=torch.bfloat16, device="cuda")
    spinf.linear(x, w_qkv, y)
    q = y[:, :Hq * d].contiguous().view(lay.T_pad, Hq, d)
    k = y[:, Hq * d:(Hq + Hkv) * d].contiguous().view(lay.T_pad, Hkv, d)
    v = y[:, (Hq + Hkv) * d:].contiguous().view(lay.T_pad, Hkv, d)
    spinf.rope_tree(plan, 0, q, k, Hq, Hkv, d, 10000.0)
    o = run_attention(spinf, plan, 0, q, k, v, shape)
    out = torch.empty(lay.T_pad, D, dtype=torch.bfloat16, device="cuda")
    spinf.linear(o.view(lay.T_pad, Hq * d), w_o, out)
    plan.device_status()
    rows = list(range(lay.T))
    ref = ol.packed_layer_rows(lay, x.float().cpu().numpy(), w_qkv.float().cpu().numpy(), w_o.float().cpu().numpy(),
                               Hq, Hkv, d, 10000.0, rows)
    got = out[:lay.T].float().cpu().numpy()
    assert np.abs(got - ref).max() <= 5e-2
