"""Pins of the oracle scoring and of the e4m3 format.

* lse and token log-probs against scipy's log-softmax on the full logits;
* a zero lm-head gives ``lse = log V`` and ``lp = -log V`` per token;
* e4m3 decode/encode against torch's float8_e4m3fn (a library routine);
* fp8 scoring: quantised weights and rows rebuilt with torch agree with the oracle.
"""
import numpy as np
import torch
from scipy.special import log_softmax, logsumexp

from oracle import fp8
from oracle import score as osc


def _data(M=6, V=1024, D=256, seed=0):
    g = np.random.default_rng(seed)
    h = torch.from_numpy(g.standard_normal((M, D), dtype=np.float32)).to(torch.bfloat16).float().numpy()
    w = torch.from_numpy((g.standard_normal((V, D), dtype=np.float32) / 16)).to(torch.bfloat16).float().numpy()
    gm = np.repeat(np.arange(M), 2)
    gt = g.integers(0, V, size=2 * M)
    return h, w, gm, gt


def test_lse_and_token_lp_match_scipy_log_softmax():
    h, w, gm, gt = _data()
    lse, lp = osc.score_rows(h, gm, gt, w=w, chunk=300)
    z = h.astype(np.float64) @ w.astype(np.float64).T
    np.testing.assert_allclose(lse, logsumexp(z, axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp, log_softmax(z, axis=1)[gm, gt], rtol=0, atol=1e-12)


def test_zero_weights_give_uniform_distribution():
    h, w, gm, gt = _data()
    lse, lp = osc.score_rows(h, gm, gt, w=np.zeros_like(w))
    np.testing.assert_allclose(lse, np.log(w.shape[0]), atol=1e-12)
    np.testing.assert_allclose(lp, -np.log(w.shape[0]), atol=1e-12)


def test_token_lp_is_a_log_probability():
    h, w, _, _ = _data(M=3, V=257)
    gm = np.repeat(np.arange(3), 257)
    gt = np.tile(np.arange(257), 3)
    _, lp = osc.score_rows(h, gm, gt, w=w, chunk=100)
    np.testing.assert_allclose(np.exp(lp).reshape(3, 257).sum(1), 1.0, atol=1e-12)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8.decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    assert fp8.decode(np.uint8(0x7E)) == 448.0 and fp8.decode(np.uint8(1)) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * 50,
        g.standard_normal(5000).astype(np.float32) * 1e-2,
        fp8.decode(np.arange(127, dtype=np.uint8)).astype(np.float32),
        # exact midpoints between neighbours: ties to even
        ((fp8.decode(np.arange(126, dtype=np.uint8)) + fp8.decode(np.arange(1, 127, dtype=np.uint8))) / 2).astype(np.float32),
        -np.float32([0.0, 1e-30, 2.0 ** -10, 3 * 2.0 ** -10]),
    ])
    vals = np.clip(vals, -448, 448).astype(np.float32)
    ours = fp8.encode_rne_sat(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)
    assert fp8.encode_rne_sat(np.float32(1e6)) == 0x7E
    assert fp8.encode_rne_sat(np.float32(-1e6)) == 0xFE


def test_quantize_rows_matches_torch_recipe():
    g = np.random.default_rng(2)
    x = torch.from_numpy(g.standard_normal((7, 300), dtype=np.float32)).to(torch.bfloat16).float()
    x[3] = 0
    codes, s = fp8.quantize_rows(x.numpy())
    absmax = x.abs().amax(1)
    ts = torch.where(absmax == 0, torch.ones_like(absmax), absmax / 448.0)
    tc = (x / ts[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    np.testing.assert_array_equal(s, ts.numpy())
    np.testing.assert_array_equal(codes, tc.numpy())


def test_fp8_scoring_uses_dequantised_operands():
    h, w, gm, gt = _data(M=4, V=300, D=128)
    wc, ws = fp8.quantize_rows(w)
    lse, lp = osc.score_rows(h, gm, gt, w_codes=wc, w_scale=ws, chunk=77)
    hc, hs = fp8.quantize_rows(h)
    hq = torch.from_numpy(hc).view(torch.float8_e4m3fn).double().numpy() * hs[:, None]
    wq = torch.from_numpy(wc).view(torch.float8_e4m3fn).double().numpy() * ws[:, None]
    z = hq @ wq.T
    np.testing.assert_allclose(lse, logsumexp(z, axis=1), atol=1e-12)
    np.testing.assert_allclose(lp, log_softmax(z, axis=1)[gm, gt], atol=1e-12)
    # and the quantisation moves the answer only a little
    lse_b, _ = osc.score_rows(h, gm, gt, w=w)
    assert np.max(np.abs(lse_b - lse)) < 0.1
