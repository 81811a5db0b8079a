"""Shared helpers of the GPU parity tests (inputs from synth, layouts from the oracle)."""
import numpy as np
import torch

from oracle import plan as op
from synth import values as sv


def pass_values(lay, shape, device="cuda", hidden_rows=True):
    """bf16 q, k, v (and hidden at the scoring rows) of one laid-out pass, on the device."""
    keys = sv.path_keys(lay.tok, lay.parent, lay.T)
    q, k, v = sv.qkv(keys, lay.T_pad, shape.n_q_heads, shape.n_kv_heads, shape.d_head)
    h = None
    if hidden_rows:
        h = sv.hidden(keys, lay.T_pad, shape.d_model, rows=lay.slot_row.tolist())
    dev = lambda t: None if t is None else t.to(device)  # noqa: E731
    return dev(q), dev(k), dev(v), dev(h)


def run_attention(spinf, plan, p, q, k, v, shape, window=0):
    o = torch.full_like(q, float("nan"))
    plan.upload(p)
    spinf.branch_attention(plan, p, q, k, v, o, shape.n_q_heads, shape.n_kv_heads, shape.d_head, window=window)
    plan.device_status()
    torch.cuda.synchronize()
    return o


def run_score(spinf, plan, p, hidden, w, w_scale, w_dtype, shape):
    info = plan.pass_info(p)
    plan.upload(p)
    nbytes = spinf.score_workspace_bytes(plan, p, shape.vocab, shape.d_model, w_dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lse = torch.full((max(info.M, 1),), float("nan"), device="cuda")
    tlp = torch.full((max(info.G, 1),), float("nan"), device="cuda")
    spinf.score(plan, p, hidden, w, w_scale, w_dtype, shape.d_model, shape.vocab, lse, tlp, ws)
    plan.device_status()
    torch.cuda.synchronize()
    return lse[:info.M].cpu().numpy(), tlp[:info.G].cpu().numpy(), ws


def oracle_plan(inputs, **kw):
    return op.plan(inputs, **kw)


def real_rows(lay):
    return np.arange(lay.T)


def sample_rows(lay, n, seed):
    """At least ``n`` rows of a laid-out pass (every row when the pass is smaller): an equal
    share drawn from every laid-out input (user chunks and floors), each input's first and
    last rows, a spread of the scoring rows, then rows drawn from the rest up to ``n``."""
    g = np.random.default_rng(seed)
    starts = [u.start for u in lay.units] + [lay.T]
    per = -(-n // max(1, len(lay.units)))
    rows = set()
    for a, b in zip(starts, starts[1:]):
        if b > a:
            rows |= set(g.choice(np.arange(a, b), size=min(per, b - a), replace=False).tolist())
            rows |= {a, b - 1}
    rows |= set(lay.slot_row[:: max(1, len(lay.slot_row) // 64)].tolist())
    if len(rows) < n:   # small inputs (floors) could not fill their share: top up from the rest
        rest = np.setdiff1d(np.arange(lay.T), np.fromiter(rows, dtype=np.int64))
        rows |= set(g.choice(rest, size=min(n - len(rows), len(rest)), replace=False).tolist())
    return sorted(int(r) for r in rows)


def pack_token_sets(sets):
    """Boolean ``[n_sets, V]`` allowed-token sets as the ABI's bitmasks: int32
    ``[n_sets, ceil(V / 32)]``, bit ``v % 32`` of word ``v // 32`` for token ``v``."""
    sets = np.asarray(sets, dtype=bool)
    n, V = sets.shape
    padded = np.zeros((n, -(-V // 32) * 32), dtype=bool)
    padded[:, :V] = sets
    words = np.packbits(padded.reshape(n, -1, 8), axis=2, bitorder="little").reshape(n, -1).view("<u4")
    return torch.from_numpy(words.view(np.int32).copy())


def run_score_extract(spinf, plan, p, hidden, w, w_scale, w_dtype, shape, sets=None, k=None):
    """spinf_score_extract on one pass: (lse, token lps, top tokens [X, k], top lps [X, k])."""
    info = plan.pass_info(p)
    k = k if k is not None else plan.extract_counts()[1]
    plan.upload(p)
    nbytes = spinf.score_workspace_bytes(plan, p, shape.vocab, shape.d_model, w_dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lse = torch.full((max(info.M, 1),), float("nan"), device="cuda")
    tlp = torch.full((max(info.G, 1),), float("nan"), device="cuda")
    top_tok = torch.full((max(info.X, 1), k), -7, dtype=torch.int32, device="cuda")
    top_lp = torch.full((max(info.X, 1), k), float("nan"), device="cuda")
    ex = {"top_tok": top_tok, "top_lp": top_lp,
          "token_sets": None if sets is None else pack_token_sets(sets).cuda()}
    spinf.score(plan, p, hidden, w, w_scale, w_dtype, shape.d_model, shape.vocab, lse, tlp, ws, extract=ex)
    plan.device_status()
    torch.cuda.synchronize()
    return (lse[:info.M].cpu().numpy(), tlp[:info.G].cpu().numpy(), top_tok[:info.X].cpu().numpy(),
            top_lp[:info.X].cpu().numpy())
