"""The oracle's pins catch the mistakes one could plausibly make in it.

Each case plants one mistake in a copy of an oracle module (a wrong scale or head
map, an off-by-one, a dropped term or factor, swapped operands, another tie or
order rule), runs that module's pins against the copy in a fresh interpreter, and
expects at least one pin to fail.  The product is not involved.  Two mistakes are
left out on purpose, being no mistakes: dropping e4m3's explicit saturation (the
nearest-code search is already bounded by the largest finite code), and sending an
input of exactly the budget through the split path (the greedy split then keeps all
of its questions in one unit, the same unit).
"""
import concurrent.futures
import json
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

PINS = {
    "attention": ["test_oracle_attention.py"],
    "score": ["test_oracle_score.py", "test_oracle_extract.py"],
    "collect": ["test_oracle_collect.py", "test_oracle_extract.py"],
    "decode": ["test_oracle_decode.py"],
    "fp8": ["test_oracle_score.py", "test_oracle_layer.py"],
    "layer": ["test_oracle_layer.py"],
    "plan": ["test_oracle_plan.py", "test_oracle_grid.py", "test_oracle_extract.py"],
}

MUTANTS = [
    ("attention-scale", "attention", "scale = 1.0 / math.sqrt(d)", "scale = 1.0 / d"),
    ("attention-head-map", "attention", "g = h * n_kv_heads // n_q_heads", "g = h % n_kv_heads"),
    ("attention-window", "attention", "layout.pos[row] - layout.pos[keys] < window",
     "layout.pos[row] - layout.pos[keys] <= window"),
    ("attention-no-normalisation", "attention", "out[i, h] = (w @ vv) / w.sum()", "out[i, h] = (w @ vv)"),
    ("attention-k-for-v", "attention", "vv = np.asarray(v[keys, g], dtype=np.float64)",
     "vv = np.asarray(k[keys, g], dtype=np.float64)"),
    ("lse-without-max", "score", "(m + np.log(np.sum(np.exp(z - m)", "(np.log(np.sum(np.exp(z - m)"),
    ("token-lp-sign", "score", "return lse, z[gm, gt] - lse[gm]", "return lse, lse[gm] - z[gm, gt]"),
    ("weight-scale-dropped", "score",
     "return fp8.decode(w_codes[rows]) * np.asarray(w_scale[rows], dtype=np.float64)[:, None]",
     "return fp8.decode(w_codes[rows])"),
    ("activation-scale-dropped", "score", "return fp8.decode(codes) * s.astype(np.float64)[:, None]",
     "return fp8.decode(codes)"),
    ("topk-ties-by-higher-id", "score", "order = np.lexsort((cand, -z_row[cand]))",
     "order = np.lexsort((-cand, -z_row[cand]))"),
    ("topk-lp-without-lse", "score", "lp[:len(top)] = z_row[top] - lse_row", "lp[:len(top)] = z_row[top]"),
    ("p-not-renormalised", "collect", "p = e / e.sum()", "p = e"),
    ("residual-sign", "collect", "residual = -np.expm1(m + np.log(e.sum()))",
     "residual = np.expm1(m + np.log(e.sum()))"),
    ("option-lp-last-token-only", "collect", "acc += float(tl[g])", "acc = float(tl[g])"),
    ("extract-answer-by-question-index", "collect", "x = plan.passes[p].questions[idx].extract", "x = j"),
    ("decode-without-anchor", "decode", "pk = np.asarray(layout.visible(int(anchor[r])), dtype=np.int64)",
     "pk = np.asarray(layout.visible(int(anchor[r]))[:-1], dtype=np.int64)"),
    ("decode-without-self", "decode", "ck = np.asarray(chain(parent, r), dtype=np.int64)",
     "ck = np.asarray(chain(parent, r)[:-1], dtype=np.int64)"),
    ("decode-head-map", "decode", "g = h * n_kv_heads // n_q_heads", "g = h % n_kv_heads"),
    ("decode-chain-order", "decode", "return out[::-1]", "return out"),
    ("e4m3-subnormal-step", "fp8", "val = np.where(e == 0, m * 2.0 ** -9,", "val = np.where(e == 0, m * 2.0 ** -10,"),
    ("e4m3-ties-down", "fp8", "pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))", "pick_lo = (d_lo <= d_hi)"),
    ("e4m3-row-scale", "fp8", "scale = (absmax / np.float32(448.0)).astype(np.float32)",
     "scale = (absmax / np.float32(240.0)).astype(np.float32)"),
    ("static-scale-multiplied", "layer",
     "scaled = (np.asarray(x, dtype=np.float32) / np.float32(x_scale)).astype(np.float32)",
     "scaled = (np.asarray(x, dtype=np.float32) * np.float32(x_scale)).astype(np.float32)"),
    ("fp8-linear-x-scale-dropped", "layer", "xs = fp8.decode(x_codes) * float(np.float32(x_scale))",
     "xs = fp8.decode(x_codes)"),
    ("qkv-k-v-swapped", "layer",
     "y[:, nq:nq + nk].reshape(T, n_kv_heads, d_head),\n            y[:, nq + nk:nq + 2 * nk].reshape(T, n_kv_heads, d_head))",
     "y[:, nq + nk:nq + 2 * nk].reshape(T, n_kv_heads, d_head),\n            y[:, nq:nq + nk].reshape(T, n_kv_heads, d_head))"),
    ("qkv-k-not-turned", "layer", "return rope(q, pos, theta), rope(k, pos, theta), v",
     "return rope(q, pos, theta), k, v"),
    ("rope-exponent", "layer", "inv_freq = float(theta) ** (-2.0 * np.arange(half) / d)",
     "inv_freq = float(theta) ** (-1.0 * np.arange(half) / d)"),
    ("rope-interleaved-pairs", "layer", "x0, x1 = x[..., :half], x[..., half:]",
     "x0, x1 = x[..., 0::2], x[..., 1::2]"),
    ("rope-turn-reversed", "layer", "return np.concatenate([x0 * c - x1 * s, x1 * c + x0 * s], axis=-1)",
     "return np.concatenate([x0 * c + x1 * s, x1 * c - x0 * s], axis=-1)"),
    ("pack-exact-fit-splits", "plan", "if cur and total + u.size > budget:", "if cur and total + u.size >= budget:"),
    ("pos-off-by-one", "plan", "pos = [content_hi[q] - content_lo[q] + len(chain[q]) - 1 for q in range(T)]",
     "pos = [content_hi[q] - content_lo[q] + len(chain[q]) for q in range(T)]"),
    ("option-token-wrong-row", "plan", "gather_rows.append(node_row[tuple(opt[:i])])",
     "gather_rows.append(node_row[tuple(opt[:max(i - 1, 0)])])"),
    ("content-end-off-by-one", "plan", "end[s + c - 1] = max(end[s + c - 1], run + 1)",
     "end[s + c - 1] = max(end[s + c - 1], run)"),
    ("tile-len-past-input", "plan", "tile_len.append(min(TILE, e - (s + TILE * j)))", "tile_len.append(TILE)"),
    ("template-sees-no-template", "plan", "chain.append((chain[prev] if prev >= s + L else []) + [r])",
     "chain.append([r])"),
    ("trie-node-under-slot", "plan", "p = node_row[prefix[:-1]]", "p = slot"),
    ("schedule-drops-last-content-tile", "plan", "hit.update(range(0, (content_hi[q] - 1 - s) // TILE + 1))",
     "hit.update(range(0, (content_hi[q] - 1 - s) // TILE))"),
    ("trie-children-sorted", "plan", "for t, child in node.items():", "for t, child in sorted(node.items()):"),
    ("grid-first-placeholder-fastest", "plan", "for combo in itertools.product(*values):",
     "for combo in (c[::-1] for c in itertools.product(*values[::-1])):"),
    ("grid-value-after-segment", "plan", "template += list(value) + list(seg)", "template += list(seg) + list(value)"),
    ("template-misses-last-content-row", "plan",
     "                parent.append(prev)\n                content_lo.append(s)\n                content_hi.append(s + L)",
     "                parent.append(prev)\n                content_lo.append(s)\n                content_hi.append(s + L - 1)"),
    ("searched-slot-wrong-row", "plan", "x_rows.append(slot)", "x_rows.append(slot - 1)"),
    ("allowed-set-ignored", "score", "toks[x], lps[x] = topk_allowed(z[x], lse[x], None if s < 0 else token_sets[s], k)",
     "toks[x], lps[x] = topk_allowed(z[x], lse[x], None, k)"),
    ("topk-one-short", "score", "top = cand[order[:k]]", "top = cand[order[:k - 1]]"),
    ("floor-is-the-question-itself", "collect", "flp = question_lp(plan.floor_home[key])", "flp = question_lp(home)"),
    ("content-limit-exclusive", "plan", 'if len(content) > o["max_content_tokens"]:',
     'if len(content) >= o["max_content_tokens"]:'),
    ("template-limit-exclusive", "plan", 'if len(template) > o["max_query_tokens"]:',
     'if len(template) >= o["max_query_tokens"]:'),
    ("options-limit-exclusive", "plan", 'if len(options) > o["max_options"]:', 'if len(options) >= o["max_options"]:'),
    ("option-tokens-limit-exclusive", "plan", 'if len(opt) > o["max_option_tokens"]:',
     'if len(opt) >= o["max_option_tokens"]:'),
    ("split-prefix-exclusive", "plan", "while j < len(questions) and size + sizes[j] <= budget:",
     "while j < len(questions) and size + sizes[j] < budget:"),
    ("floor-prefix-ignored", "plan", '        prefix = tuple(o["floor_prefix"])', "        prefix = ()"),
    ("floors-in-reverse-order", "plan",
     "        for content, questions in inputs:\n            for question in questions:\n                if is_searched",
     "        for content, questions in inputs[::-1]:\n            for question in questions:\n                if is_searched"),
    ("floor-budget-exclusive", "plan", "                if size > budget:\n                    raise PlanError(\"LIMIT\", \"a floor",
     "                if size >= budget:\n                    raise PlanError(\"LIMIT\", \"a floor"),
]


def _run(module, old, new):
    env = dict(os.environ, ORACLE_MUTANT=json.dumps([module, old, new]),
               PYTHONPATH=os.pathsep.join([HERE, ROOT, os.environ.get("PYTHONPATH", "")]))
    files = [os.path.join(HERE, f) for f in PINS[module]]
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-q", "-x", "-m", "not gpu", "-p", "oracle_mutant_plugin",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout + r.stderr


@pytest.fixture(scope="module")
def outcomes():
    """Every mutant's pin run, several at a time (each is its own interpreter)."""
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with concurrent.futures.ThreadPoolExecutor(workers) as pool:
        futures = {m[0]: pool.submit(_run, *m[1:]) for m in MUTANTS}
        return {name: f.result() for name, f in futures.items()}


@pytest.mark.parametrize("name,module,new", [(m[0], m[1], m[3]) for m in MUTANTS], ids=[m[0] for m in MUTANTS])
def test_a_planted_mistake_fails_a_pin(outcomes, name, module, new):
    code, out = outcomes[name]
    assert "mutant pattern occurs" not in out, out[-1500:]
    assert code == 1, f"no pin of oracle/{module}.py caught {new!r} (pytest exit {code}):\n{out[-1500:]}"
