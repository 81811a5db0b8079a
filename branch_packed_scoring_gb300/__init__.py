"""Python binding of the branch-packed scoring C ABI (``include/spinf.h``).

Argument marshalling only: every step of the path runs in ``libspinf.so``
(host planner and collect in C++, attention and scoring in sm_103a kernels).
There is no fallback: if the library is missing, every call raises.

Device tensors are passed as ``torch.Tensor`` (or raw integer addresses);
torch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import itertools
import os
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspinf.so")

OK, E_INVALID, E_LIMIT, E_NOMEM, E_CUDA, E_UNSUPPORTED, E_DEVICE_TIMEOUT, E_DEVICE_CHECK = range(8)
STATUS_NAMES = {0: "OK", 1: "INVALID", 2: "LIMIT", 3: "NOMEM", 4: "CUDA", 5: "UNSUPPORTED",
                6: "DEVICE_TIMEOUT", 7: "DEVICE_CHECK"}
DTYPE_BF16, DTYPE_E4M3 = 0, 1
HIDDEN_PASS_ROWS, HIDDEN_SLOT_ROWS = 0, 1
Q_SCORED, Q_SEARCHED = 0, 1

#: every symbol the header declares
SYMBOLS = [
    "spinf_plan_opts_default", "spinf_pack_plan", "spinf_plan_num_passes", "spinf_plan_pass_info",
    "spinf_plan_counts", "spinf_plan_extract_counts", "spinf_plan_upload", "spinf_plan_descriptor_bytes", "spinf_plan_upload_to",
    "spinf_plan_upload_pinned",
    "spinf_plan_window_schedule", "spinf_plan_tile_schedule", "spinf_plan_tile_schedule_q",
    "spinf_branch_attention", "spinf_score_workspace_bytes",
    "spinf_score", "spinf_score_extract", "spinf_score_static", "spinf_score_passes_workspace_bytes",
    "spinf_score_passes", "spinf_collect", "spinf_collect_extract",
    "spinf_device_status", "spinf_device_selftest",
    "spinf_rope_tree", "spinf_linear", "spinf_qkv_rope", "spinf_quantize_static",
    "spinf_decode_attention", "spinf_score_rows_workspace_bytes", "spinf_score_rows",
    "spinf_plan_free", "spinf_fingerprint",
    "spinf_status_string", "spinf_last_error",
]


class SpinfError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))


class _Tokens(ctypes.Structure):
    _fields_ = [("ids", ctypes.c_void_p), ("n", ctypes.c_int32)]


class _Opts(ctypes.Structure):
    _fields_ = [("token_budget", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("max_content_tokens", ctypes.c_int32), ("max_query_tokens", ctypes.c_int32),
                ("max_options", ctypes.c_int32), ("max_option_tokens", ctypes.c_int32),
                ("max_prompts_per_input", ctypes.c_int32), ("floors", ctypes.c_int32),
                ("floor_prefix", _Tokens), ("vocab", ctypes.c_int32), ("extract_k", ctypes.c_int32)]


_P = ctypes.POINTER(ctypes.c_int32)


class _PassInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "T_pad", "n_qtiles", "n_sched", "M", "G", "n_units")] + \
               [(n, _P) for n in ("tok", "parent", "pos", "end", "anchor", "tile_ptr", "tile_kv", "tile_len", "slot_row",
                                  "gather_m", "gather_tok", "unit_start", "unit_source", "row_runs")] + \
               [("X", ctypes.c_int32), ("x_m", _P), ("x_set", _P)]


_D = ctypes.POINTER(ctypes.c_double)


class _ExtractOut(ctypes.Structure):
    _fields_ = [("token_sets", ctypes.c_void_p), ("n_sets", ctypes.c_int32), ("top_tok", ctypes.c_void_p),
                ("top_lp", ctypes.c_void_p)]


class _Result(ctypes.Structure):
    _fields_ = [(n, _D) for n in ("option_lp", "option_p", "option_floor_lp", "option_floor_p", "residual",
                                  "floor_residual")]


# numpy views of the request structs (same layout as the header on LP64)
_TOK = np.dtype([("ids", "<u8"), ("n", "<i4"), ("_pad", "<i4")])
_QUE = np.dtype([("tmpl_ids", "<u8"), ("tmpl_n", "<i4"), ("_p0", "<i4"), ("options", "<u8"),
                 ("n_options", "<i4"), ("kind", "<i4"), ("token_set", "<i4"), ("_p1", "<i4")])
_INP = np.dtype([("content_ids", "<u8"), ("content_n", "<i4"), ("_p0", "<i4"), ("questions", "<u8"),
                 ("n_questions", "<i4"), ("_p1", "<i4"), ("grids", "<u8"), ("n_grids", "<i4"), ("_p2", "<i4")])
_GRID = np.dtype([("segments", "<u8"), ("n_placeholders", "<i4"), ("_p0", "<i4"), ("values", "<u8"),
                  ("n_values", "<u8"), ("options", "<u8"), ("n_options", "<i4"), ("kind", "<i4"),
                  ("token_set", "<i4"), ("_p1", "<i4")])

_lib = None


def lib():
    """The loaded ``libspinf.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m branch_packed_scoring_gb300.build` "
                           "(or __graft_entry__.build()); there is no fallback implementation")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.spinf_plan_opts_default.argtypes = [ctypes.POINTER(_Opts)]
    L.spinf_plan_opts_default.restype = None
    L.spinf_pack_plan.argtypes = [vp, i32, ctypes.POINTER(_Opts), ctypes.POINTER(vp)]
    L.spinf_plan_num_passes.argtypes = [vp]
    L.spinf_plan_num_passes.restype = i32
    L.spinf_plan_pass_info.argtypes = [vp, i32, ctypes.POINTER(_PassInfo)]
    L.spinf_plan_counts.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.spinf_plan_extract_counts.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i32)]
    L.spinf_plan_upload.argtypes = [vp, i32, vp]
    L.spinf_plan_descriptor_bytes.argtypes = [vp, i32]
    L.spinf_plan_descriptor_bytes.restype = sz
    L.spinf_plan_upload_to.argtypes = [vp, i32, vp, sz, vp]
    L.spinf_plan_upload_pinned.argtypes = [vp, i32, vp, sz, vp, sz, vp]
    L.spinf_plan_window_schedule.argtypes = [vp, i32, i32, ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                                             ctypes.POINTER(i32)]
    L.spinf_plan_tile_schedule_q.argtypes = [vp, i32, i32, i32, i32, ctypes.POINTER(_P), ctypes.POINTER(_P),
                                             ctypes.POINTER(_P), ctypes.POINTER(i32)]
    L.spinf_plan_tile_schedule.argtypes = [vp, i32, i32, i32, ctypes.POINTER(_P), ctypes.POINTER(_P),
                                           ctypes.POINTER(_P), ctypes.POINTER(i32)]
    L.spinf_branch_attention.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, f32, i32, vp]
    L.spinf_score_workspace_bytes.argtypes = [vp, i32, i32, i32, i32]
    L.spinf_score_workspace_bytes.restype = sz
    L.spinf_score.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spinf_score_extract.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, vp, vp, ctypes.POINTER(_ExtractOut), vp,
                                      sz, vp]
    L.spinf_score_static.argtypes = [vp, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp]
    L.spinf_score_passes_workspace_bytes.argtypes = [vp, i32, vp, i32, i32, i32]
    L.spinf_score_passes_workspace_bytes.restype = sz
    L.spinf_score_passes.argtypes = [vp, i32, vp, vp, i32, vp, vp, i32, i32, i32, vp, vp, vp, sz, vp]
    L.spinf_collect.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(_Result)]
    L.spinf_collect_extract.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp]
    L.spinf_device_status.argtypes = [vp, vp]
    L.spinf_device_selftest.argtypes = [vp, i32, vp]
    L.spinf_rope_tree.argtypes = [vp, i32, vp, vp, i32, i32, i32, f32, vp]
    L.spinf_linear.argtypes = [vp, vp, vp, vp, f32, i32, vp, i64, i64, i64, vp]
    L.spinf_qkv_rope.argtypes = [vp, i32, vp, vp, vp, f32, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp]
    L.spinf_quantize_static.argtypes = [vp, f32, vp, i64, vp]
    L.spinf_decode_attention.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, i32, vp, i32, i32, i32, f32,
                                         vp]
    L.spinf_score_rows_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.spinf_score_rows_workspace_bytes.restype = sz
    L.spinf_score_rows.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, vp, vp, i32, i32, vp, vp, vp, vp, sz, vp]
    L.spinf_plan_free.argtypes = [vp]
    L.spinf_plan_free.restype = None
    L.spinf_fingerprint.restype = ctypes.c_char_p
    L.spinf_status_string.argtypes = [i32]
    L.spinf_status_string.restype = ctypes.c_char_p
    L.spinf_last_error.restype = ctypes.c_char_p
    for name in ("spinf_pack_plan", "spinf_plan_pass_info", "spinf_plan_counts", "spinf_plan_extract_counts",
                 "spinf_plan_upload", "spinf_plan_upload_to", "spinf_plan_upload_pinned", "spinf_plan_window_schedule", "spinf_plan_tile_schedule",
                 "spinf_plan_tile_schedule_q",
                 "spinf_branch_attention", "spinf_score", "spinf_score_extract", "spinf_score_static",
                 "spinf_score_passes", "spinf_collect",
                 "spinf_collect_extract",
                 "spinf_device_status", "spinf_device_selftest", "spinf_rope_tree", "spinf_linear",
                 "spinf_qkv_rope", "spinf_quantize_static", "spinf_decode_attention", "spinf_score_rows"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def _check(status):
    if status != OK:
        raise SpinfError(status, lib().spinf_last_error().decode())


def _ptr(x):
    """Device/host address of a torch tensor, numpy array or int (None -> 0)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_KINDS = None


def _kinds():
    global _KINDS
    if _KINDS is None:
        import torch
        words = (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ())
        _KINDS = {"bf16": (torch.bfloat16,), "f32": (torch.float32,), "i32": (torch.int32,),
                  "e4m3": (torch.uint8, torch.float8_e4m3fn), "words": words, "bytes": None}
    return _KINDS


def _wkind(w_dtype):
    return "e4m3" if w_dtype == DTYPE_E4M3 else "bf16" if w_dtype == DTYPE_BF16 else "bytes"


class _Args:
    """The device-buffer arguments of one call, checked before the C call.  A torch tensor
    must have the dtype the header gives, be contiguous, hold at least the elements the call
    reads or writes, and live on the current CUDA device; otherwise SpinfError(INVALID).  A
    raw device address (int) or None passes unchecked, as it would through the C ABI."""

    def __init__(self, call):
        self.call = call
        self.device = None

    def bad(self, msg):
        raise SpinfError(E_INVALID, f"{self.call}: {msg}")

    def __call__(self, x, what, kind, n=None):
        if x is None or isinstance(x, int):
            return x
        if not hasattr(x, "is_cuda"):
            self.bad(f"{what} must be a torch tensor or a device address, not {type(x).__name__}")
        dts = _kinds()[kind]
        if dts is not None and x.dtype not in dts:
            self.bad(f"{what} has dtype {x.dtype}; {kind} expected")
        if not x.is_contiguous():
            self.bad(f"{what} must be contiguous")
        if n is not None and x.numel() < n:
            self.bad(f"{what} holds {x.numel()} elements; the call needs {n}")
        if not x.is_cuda:
            self.bad(f"{what} must be a CUDA tensor (it is on {x.device})")
        if self.device is None:
            import torch
            self.device = torch.cuda.current_device()
        if x.device.index != self.device:
            self.bad(f"{what} is on {x.device}; the current device is cuda:{self.device}")
        return x.data_ptr()


def fingerprint() -> str:
    return lib().spinf_fingerprint().decode()


@dataclass
class PassInfo:
    T: int
    T_pad: int
    n_qtiles: int
    n_sched: int
    M: int
    G: int
    n_units: int
    tok: np.ndarray
    parent: np.ndarray
    pos: np.ndarray
    end: np.ndarray
    anchor: np.ndarray
    tile_ptr: np.ndarray
    tile_kv: np.ndarray
    tile_len: np.ndarray
    slot_row: np.ndarray
    gather_m: np.ndarray
    gather_tok: np.ndarray
    unit_start: np.ndarray
    unit_source: np.ndarray
    row_runs: np.ndarray
    X: int = 0
    x_m: np.ndarray = None
    x_set: np.ndarray = None


def _marshal(inputs):
    """Lay the request out as the header's structs in numpy buffers (kept alive by the caller).

    Every token array is one (pointer, length) pair into a single int32 buffer; a sequence
    object that recurs in the request is stored once.  Inputs that share one question-list
    object (the same question set asked of many contents) share one array of question
    structs, so each distinct list is walked once."""
    block_of, blocks, in_block, grids = {}, [], [], []
    for i, inp in enumerate(inputs):
        qs = inp[1]
        b = block_of.setdefault(id(qs), len(blocks))
        if b == len(blocks):
            blocks.append(qs)
        in_block.append(b)
        if len(inp) > 2:
            grids.extend((i, g) for g in inp[2])
    seqs = [inp[0] for inp in inputs]   # the contents, then each block's templates and options
    kind, tset, n_opt, block_q0 = [], [], [], []
    for qs in blocks:
        block_q0.append(len(n_opt))
        for question in qs:
            seqs.append(question[0])
            options = question[1]
            if options is None and len(question) == 3:   # searched slot: (template, None, token_set)
                kind.append(Q_SEARCHED)
                tset.append(int(question[2]))
                n_opt.append(0)
            else:
                kind.append(Q_SCORED)
                tset.append(-1)
                n_opt.append(len(options))
                seqs.extend(options)
    # one stored copy per distinct sequence object
    slot_of, uniq = {}, []
    where = np.empty(len(seqs), dtype=np.int64)
    for s, seq in enumerate(seqs):
        u = slot_of.setdefault(id(seq), len(uniq))
        if u == len(uniq):
            uniq.append(seq)
        where[s] = u
    ulen = np.fromiter(map(len, uniq), dtype=np.int64, count=len(uniq))
    uoff = np.zeros(len(uniq) + 1, dtype=np.int64)
    np.cumsum(ulen, out=uoff[1:])
    total = int(uoff[-1])
    flat = (np.fromiter(itertools.chain.from_iterable(uniq), dtype=np.int32, count=total) if total
            else np.zeros(1, dtype=np.int32))
    lens = ulen[where]
    addr = np.where(lens > 0, np.uint64(flat.ctypes.data) + np.uint64(4) * uoff[:-1][where].astype(np.uint64),
                    np.uint64(0))
    n_in, nt = len(inputs), len(n_opt)
    n_opt_arr = np.asarray(n_opt, dtype=np.int64)
    q_first = np.zeros(nt + 1, dtype=np.int64)
    np.cumsum(1 + n_opt_arr, out=q_first[1:])
    t_idx = n_in + q_first[:-1]                                 # each question's template
    o_mask = np.ones(len(seqs) - n_in, dtype=bool)
    o_mask[q_first[:-1]] = False
    o_idx = n_in + np.flatnonzero(o_mask)                       # options, question by question
    tok = np.zeros(max(len(o_idx), 1), dtype=_TOK)
    que = np.zeros(max(nt, 1), dtype=_QUE)
    inp = np.zeros(n_in, dtype=_INP)
    if len(o_idx):
        tok["ids"][:len(o_idx)] = addr[o_idx]
        tok["n"][:len(o_idx)] = lens[o_idx]
    if nt:
        que["tmpl_ids"][:nt] = addr[t_idx]
        que["tmpl_n"][:nt] = lens[t_idx]
        first_opt = np.concatenate([[0], np.cumsum(n_opt_arr)[:-1]]).astype(np.uint64)
        que["options"][:nt] = np.uint64(tok.ctypes.data) + np.uint64(_TOK.itemsize) * first_opt
        que["n_options"][:nt] = n_opt_arr
        que["kind"][:nt] = kind
        que["token_set"][:nt] = tset
    if n_in:
        inp["content_ids"] = addr[:n_in]
        inp["content_n"] = lens[:n_in]
        bq = np.asarray([len(qs) for qs in blocks], dtype=np.int64)[in_block]
        q0 = np.asarray(block_q0, dtype=np.uint64)[in_block]
        inp["questions"] = np.where(bq > 0, np.uint64(que.ctypes.data) + np.uint64(_QUE.itemsize) * q0, np.uint64(0))
        inp["n_questions"] = bq
    keep = [flat, que, tok]
    if grids:
        _marshal_grids(inp, grids, keep)
    return inp, tuple(keep)


def _marshal_grids(inp, grids, keep):
    """The inputs' placeholder grids as ``spinf_grid`` arrays (segments, values, options,
    value counts), pointed to from ``inp``; every buffer is appended to ``keep``."""
    ids, spans = [], []   # spans: (offset, n) of every token array, in the order used below

    def span(seq):
        spans.append((len(ids), len(seq)))
        ids.extend(int(t) for t in seq)

    meta = []
    for _, g in grids:
        segments, values, options = g[0], g[1], g[2]
        if len(segments) != len(values) + 1:
            raise ValueError("a grid needs one more segment than placeholders")
        s0 = len(spans)
        for seg in segments:
            span(seg)
        v0 = len(spans)
        for vals in values:
            for v in vals:
                span(v)
        o0 = len(spans)
        for opt in (options or ()):
            span(opt)
        meta.append((s0, v0, o0, [len(v) for v in values]))
    flat = np.array(ids, dtype=np.int32) if ids else np.zeros(1, dtype=np.int32)
    tok = np.zeros(max(len(spans), 1), dtype=_TOK)
    for i, (off, n) in enumerate(spans):
        tok[i]["ids"] = flat.ctypes.data + 4 * off if n else 0
        tok[i]["n"] = n
    counts = np.array([c for m in meta for c in m[3]] or [0], dtype=np.int32)
    arr = np.zeros(len(grids), dtype=_GRID)
    tb, isz, c0 = tok.ctypes.data, _TOK.itemsize, 0
    for j, ((_, g), (s0, v0, o0, nv)) in enumerate(zip(grids, meta)):
        searched = g[2] is None
        arr[j]["segments"] = tb + isz * s0
        arr[j]["n_placeholders"] = len(nv)
        arr[j]["values"] = tb + isz * v0 if nv else 0
        arr[j]["n_values"] = counts.ctypes.data + 4 * c0 if nv else 0
        arr[j]["options"] = 0 if searched else tb + isz * o0
        arr[j]["n_options"] = 0 if searched else len(g[2])
        arr[j]["kind"] = Q_SEARCHED if searched else Q_SCORED
        arr[j]["token_set"] = int(g[3]) if searched else -1
        c0 += len(nv)
    first = {}
    for j, (i, _) in enumerate(grids):
        first.setdefault(i, j)
        inp[i]["n_grids"] += 1
    for i, j in first.items():
        inp[i]["grids"] = arr.ctypes.data + _GRID.itemsize * j
    keep += [flat, tok, counts, arr]


class Request:
    """A request laid out once in the header's structs (``spinf_input`` arrays).

    Planning the same request again (``Plan(request)``) then costs only the C
    planner, not the Python marshalling of nested lists.  Marshalling is cheapest
    when inputs that ask the same questions share one question-list object: that
    list is walked once and its question structs are shared.
    """

    def __init__(self, inputs):
        self.n_inputs = len(inputs)
        self.inp, self._keep = _marshal(inputs)


class Plan:
    """A packed layout of a request (``spinf_pack_plan``).  Owns its device copies.

    ``inputs`` is a list of ``(content_ids, [question, ...])`` (optionally a third
    element, a list of placeholder grids) or a :class:`Request`; a question is
    ``(template_ids, [option_ids, ...])`` (scored) or ``(template_ids, None, token_set)``
    (a searched slot, ``token_set`` -1 for any token).  Inputs that ask the same
    questions can share one question-list object, which is then marshalled once.
    """

    def __init__(self, inputs, *, token_budget=None, max_tokens=None, max_content_tokens=None,
                 max_query_tokens=None, max_options=None, max_option_tokens=None, max_prompts_per_input=None,
                 floors=True, floor_prefix=(), vocab=0, extract_k=None):
        L = lib()
        self._h = None
        self._size_cache = {}
        opts = _Opts()
        L.spinf_plan_opts_default(ctypes.byref(opts))
        for name, val in (("token_budget", token_budget), ("max_tokens", max_tokens),
                          ("max_content_tokens", max_content_tokens), ("max_query_tokens", max_query_tokens),
                          ("max_options", max_options), ("max_option_tokens", max_option_tokens),
                          ("max_prompts_per_input", max_prompts_per_input)):
            if val is not None:
                setattr(opts, name, int(val))
        opts.floors = 1 if floors else 0
        fp = np.ascontiguousarray(np.asarray(floor_prefix, dtype=np.int32).ravel())
        opts.floor_prefix.ids = fp.ctypes.data if len(fp) else None
        opts.floor_prefix.n = len(fp)
        opts.vocab = int(vocab)
        if extract_k is not None:
            opts.extract_k = int(extract_k)
        if isinstance(inputs, Request):
            inp, keep, n_inputs = inputs.inp, None, inputs.n_inputs
        else:
            (inp, keep), n_inputs = _marshal(inputs), len(inputs)
        h = ctypes.c_void_p()
        _check(L.spinf_pack_plan(inp.ctypes.data if len(inp) else None, n_inputs, ctypes.byref(opts),
                                 ctypes.byref(h)))
        del keep, fp
        self._h = h
        self.num_passes = L.spinf_plan_num_passes(h)

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan is closed")
        return self._h

    def _sizes(self, p):
        """(T_pad, M, G, X) of pass p, without copying its arrays (cached)."""
        s = self._size_cache.get(p)
        if s is None:
            info = _PassInfo()
            _check(lib().spinf_plan_pass_info(self.handle, p, ctypes.byref(info)))
            s = self._size_cache[p] = (info.T_pad, info.M, info.G, info.X)
        return s

    def pass_info(self, p) -> PassInfo:
        info = _PassInfo()
        _check(lib().spinf_plan_pass_info(self.handle, p, ctypes.byref(info)))

        def arr(ptr, n):
            return np.ctypeslib.as_array(ptr, shape=(n,)).copy() if n > 0 else np.zeros(0, dtype=np.int32)

        return PassInfo(
            T=info.T, T_pad=info.T_pad, n_qtiles=info.n_qtiles, n_sched=info.n_sched, M=info.M, G=info.G,
            n_units=info.n_units, tok=arr(info.tok, info.T_pad), parent=arr(info.parent, info.T_pad),
            pos=arr(info.pos, info.T_pad), end=arr(info.end, info.T_pad), anchor=arr(info.anchor, info.T_pad),
            tile_ptr=arr(info.tile_ptr, info.n_qtiles + 1), tile_kv=arr(info.tile_kv, info.n_sched), tile_len=arr(info.tile_len, info.n_sched),
            slot_row=arr(info.slot_row, info.M), gather_m=arr(info.gather_m, info.G),
            gather_tok=arr(info.gather_tok, info.G), unit_start=arr(info.unit_start, info.n_units + 1),
            unit_source=arr(info.unit_source, info.n_units),
            row_runs=arr(info.row_runs, 8 * info.T_pad).reshape(info.T_pad, 8),
            X=info.X, x_m=arr(info.x_m, info.X), x_set=arr(info.x_set, info.X))

    def counts(self):
        nq, no = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().spinf_plan_counts(self.handle, ctypes.byref(nq), ctypes.byref(no)))
        return nq.value, no.value

    def extract_counts(self):
        """(searched slots over the request, extract_k)."""
        n, k = ctypes.c_int64(), ctypes.c_int32()
        _check(lib().spinf_plan_extract_counts(self.handle, ctypes.byref(n), ctypes.byref(k)))
        return n.value, k.value

    def window_schedule(self, p, window):
        """(tile_ptr, tile_kv, tile_len) of pass p's schedule for a sliding window."""
        tp, tk, tl, n = _P(), _P(), _P(), ctypes.c_int32()
        _check(lib().spinf_plan_window_schedule(self.handle, p, window, ctypes.byref(tp), ctypes.byref(tk),
                                                ctypes.byref(tl), ctypes.byref(n)))
        nq = self._sizes(p)[0] // 128   # Q tiles of the pass
        arr = lambda ptr, k: np.ctypeslib.as_array(ptr, shape=(k,)).copy() if k > 0 else np.zeros(0, np.int32)  # noqa: E731
        return arr(tp, nq + 1), arr(tk, n.value), arr(tl, n.value)

    def tile_schedule(self, p, window=0, key_tile=128, q_rows=128):
        """(tile_ptr, tile_kv, tile_len) of the schedule the attention kernel runs on pass p
        for a window (0: none) in tiles of key_tile keys (128; 64 at d_head 256) and Q tiles of
        q_rows rows (128; 64 at d_head 256 with two query heads per kv head)."""
        tp, tk, tl, n = _P(), _P(), _P(), ctypes.c_int32()
        _check(lib().spinf_plan_tile_schedule_q(self.handle, p, window, key_tile, q_rows, ctypes.byref(tp),
                                                ctypes.byref(tk), ctypes.byref(tl), ctypes.byref(n)))
        nq = self._sizes(p)[0] // q_rows   # Q tiles of the pass
        arr = lambda ptr, k: np.ctypeslib.as_array(ptr, shape=(k,)).copy() if k > 0 else np.zeros(0, np.int32)  # noqa: E731
        return arr(tp, nq + 1), arr(tk, n.value), arr(tl, n.value)

    def descriptor_bytes(self, p):
        return int(lib().spinf_plan_descriptor_bytes(self.handle, p))

    def upload(self, p, stream=None, buffer=None, staging=None):
        """Descriptors of pass p to the device: into a plan-owned allocation, or into
        `buffer` (a caller-owned uint8 device tensor of >= descriptor_bytes(p) bytes);
        with `staging` (a pinned uint8 host tensor of as many bytes) the copy is made from
        there and the call does not wait for the copy engine (spinf_plan_upload_pinned)."""
        if buffer is None:
            if staging is not None:
                raise ValueError("staging needs a caller-owned device buffer")
            _check(lib().spinf_plan_upload(self.handle, p, _stream(stream)))
            return
        addr = _Args("upload")(buffer, "buffer", "bytes")
        nbytes = buffer.numel() * buffer.element_size()
        if staging is None:
            _check(lib().spinf_plan_upload_to(self.handle, p, ctypes.c_void_p(addr), nbytes, _stream(stream)))
            return
        if staging.is_cuda or not staging.is_contiguous():
            raise ValueError("staging must be a contiguous host tensor")
        _check(lib().spinf_plan_upload_pinned(self.handle, p, ctypes.c_void_p(addr), nbytes,
                                              ctypes.c_void_p(staging.data_ptr()),
                                              staging.numel() * staging.element_size(), _stream(stream)))

    def collect(self, token_lp_per_pass):
        """Per option lp / p / floor and per question residuals from host fp32 token lps."""
        nq, no = self.counts()
        out = {k: np.full(n, np.nan) for k, n in (("option_lp", no), ("option_p", no), ("option_floor_lp", no),
                                                 ("option_floor_p", no), ("residual", nq),
                                                 ("floor_residual", nq))}
        res = _Result(*[v.ctypes.data_as(_D) for v in out.values()])
        arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in token_lp_per_pass]
        if len(arrs) != self.num_passes:
            raise ValueError("one token-lp array per pass is needed")
        ptrs = (ctypes.c_void_p * max(1, len(arrs)))(*[a.ctypes.data for a in arrs])
        _check(lib().spinf_collect(self.handle, ptrs, ctypes.byref(res)))
        return out

    def collect_extract(self, top_tok_per_pass, top_lp_per_pass):
        """Searched-slot answers in question order: (tokens [n, k] int32, lp [n, k] float64)."""
        n, k = self.extract_counts()
        tok = np.full((n, k), -1, dtype=np.int32)
        lp = np.full((n, k), -np.inf)
        if len(top_tok_per_pass) != self.num_passes or len(top_lp_per_pass) != self.num_passes:
            raise ValueError("one answer array per pass is needed")
        ta = [np.ascontiguousarray(a, dtype=np.int32) for a in top_tok_per_pass]
        la = [np.ascontiguousarray(a, dtype=np.float32) for a in top_lp_per_pass]
        tp = (ctypes.c_void_p * max(1, len(ta)))(*[a.ctypes.data for a in ta])
        lpp = (ctypes.c_void_p * max(1, len(la)))(*[a.ctypes.data for a in la])
        _check(lib().spinf_collect_extract(self.handle, tp, lpp, tok.ctypes.data, lp.ctypes.data))
        return tok, lp

    def device_status(self, stream=None):
        _check(lib().spinf_device_status(self.handle, _stream(stream)))

    def device_selftest(self, wait_ms=50, stream=None):
        """Enqueue a bounded wait that runs out (see spinf_device_selftest)."""
        _check(lib().spinf_device_selftest(self.handle, wait_ms, _stream(stream)))

    def close(self):
        if self._h is not None and _lib is not None:
            _lib.spinf_plan_free(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def branch_attention(plan, p, q, k, v, o, n_q_heads, n_kv_heads, d_head, scale=0.0, window=0, stream=None):
    """spinf_branch_attention: q, o [T_pad, Hq, d] and k, v [T_pad, Hkv, d] bf16 on the device."""
    a = _Args("branch_attention")
    T = plan._sizes(p)[0]
    nq, nkv = T * n_q_heads * d_head, T * n_kv_heads * d_head
    _check(lib().spinf_branch_attention(plan.handle, p, a(q, "q", "bf16", nq), a(k, "k", "bf16", nkv),
                                        a(v, "v", "bf16", nkv), a(o, "o", "bf16", nq), n_q_heads, n_kv_heads,
                                        d_head, float(scale), int(window), _stream(stream)))


def rope_tree(plan, p, q, k, n_q_heads, n_kv_heads, d_head, theta=10000.0, stream=None):
    """Rotary embedding in place at each row's tree depth (spinf_rope_tree)."""
    a = _Args("rope_tree")
    T = plan._sizes(p)[0]
    _check(lib().spinf_rope_tree(plan.handle, p, a(q, "q", "bf16", T * n_q_heads * d_head),
                                 a(k, "k", "bf16", T * n_kv_heads * d_head), n_q_heads, n_kv_heads, d_head,
                                 float(theta), _stream(stream)))


def linear(plan, x, w, y, w_scale=None, x_scale=1.0, w_dtype=DTYPE_BF16, stream=None):
    """y = x . w^T on the tensor cores (spinf_linear); x [rows, in], w [out, in], y [rows, out] bf16.
    With ``w_dtype=DTYPE_E4M3``, x and w are e4m3 codes (uint8), ``w_scale`` [out] fp32, ``x_scale`` static."""
    a, kind = _Args("linear"), _wkind(w_dtype)
    rows, n_in, n_out = x.shape[0], x.shape[1], w.shape[0]
    _check(lib().spinf_linear(plan.handle, a(x, "x", kind, rows * n_in), a(w, "w", kind, n_out * n_in),
                              a(w_scale, "w_scale", "f32", n_out), float(x_scale), w_dtype,
                              a(y, "y", "bf16", rows * n_out), rows, n_in, n_out, _stream(stream)))


def qkv_rope(plan, p, x, w, q, k, v, n_q_heads, n_kv_heads, d_head, theta=10000.0, w_scale=None, x_scale=1.0,
             w_dtype=DTYPE_BF16, stream=None):
    """QKV projection of pass p with the rotary turn fused (spinf_qkv_rope); writes q, k, v."""
    a, kind = _Args("qkv_rope"), _wkind(w_dtype)
    T, D = plan._sizes(p)[0], x.shape[1]
    n_qkv, nq, nkv = (n_q_heads + 2 * n_kv_heads) * d_head, T * n_q_heads * d_head, T * n_kv_heads * d_head
    _check(lib().spinf_qkv_rope(plan.handle, p, a(x, "x", kind, T * D), a(w, "w", kind, n_qkv * D),
                                a(w_scale, "w_scale", "f32", n_qkv), float(x_scale), w_dtype, D, n_q_heads,
                                n_kv_heads, d_head, float(theta), a(q, "q", "bf16", nq), a(k, "k", "bf16", nkv),
                                a(v, "v", "bf16", nkv), _stream(stream)))


def quantize_static(x, x_scale, codes, stream=None):
    """e4m3 codes of bf16 ``x`` with a static scale (spinf_quantize_static)."""
    a, n = _Args("quantize_static"), x.numel()
    _check(lib().spinf_quantize_static(a(x, "x", "bf16"), float(x_scale), a(codes, "codes", "e4m3", n), n,
                                       _stream(stream)))


def score_workspace_bytes(plan, p, vocab, d_model, w_dtype=DTYPE_BF16):
    return lib().spinf_score_workspace_bytes(plan.handle, p, vocab, d_model, w_dtype)


def score(plan, p, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp, workspace, workspace_bytes=None,
          stream=None, extract=None):
    """``spinf_score``; with ``extract`` (a dict of ``top_tok`` [X, k] int32 and ``top_lp`` [X, k] fp32 device
    tensors, optional ``token_sets`` [n_sets, ceil(vocab/32)] int32 bitmasks) ``spinf_score_extract``."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    a = _Args("score")
    args = _score_args(a, plan, p, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp)
    ws = a(workspace, "workspace", "bytes")
    if extract is None:
        _check(lib().spinf_score(plan.handle, p, *args, ws, int(workspace_bytes), _stream(stream)))
        return
    sets = extract.get("token_sets")
    n_sets = 0 if sets is None else int(sets.shape[0])
    X, k = plan._sizes(p)[3], plan.extract_counts()[1]
    ex = _ExtractOut(a(sets, "token_sets", "words", n_sets * (-(-vocab // 32))), n_sets,
                     a(extract["top_tok"], "top_tok", "i32", X * k), a(extract["top_lp"], "top_lp", "f32", X * k))
    _check(lib().spinf_score_extract(plan.handle, p, *args, ctypes.byref(ex), ws,
                                     int(workspace_bytes), _stream(stream)))


def _score_args(a, plan, p, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp):
    """Checked (hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp) of a scoring call."""
    T, M, G, _ = plan._sizes(p)
    kind = _wkind(w_dtype)
    return (a(hidden, "hidden", "bf16", T * d_model), a(w, "w", kind, vocab * d_model),
            a(w_scale, "w_scale", "f32", vocab), w_dtype, d_model, vocab, a(row_lse, "row_lse", "f32", M),
            a(token_lp, "token_lp", "f32", G))


def _pass_list(passes):
    arr = np.ascontiguousarray(np.asarray(list(passes), dtype=np.int32))
    return arr, arr.ctypes.data


def score_passes_workspace_bytes(plan, passes, vocab, d_model, w_dtype=DTYPE_BF16):
    arr, ptr = _pass_list(passes)
    return lib().spinf_score_passes_workspace_bytes(plan.handle, len(arr), ptr, vocab, d_model, w_dtype)


def score_passes(plan, passes, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp, workspace,
                 workspace_bytes=None, stream=None, slot_rows=False):
    """``spinf_score_passes``: the passes in ``passes`` scored in one sweep of the lm head; ``hidden``,
    ``row_lse`` and ``token_lp`` are lists with one device tensor per listed pass.  ``slot_rows``:
    each hidden tensor holds only its pass's scoring rows [M, d_model] (SPINF_HIDDEN_SLOT_ROWS)."""
    arr, ptr = _pass_list(passes)
    n = len(arr)
    if not (len(hidden) == len(row_lse) == len(token_lp) == n):
        raise SpinfError(E_INVALID, "score_passes: one hidden, row_lse and token_lp per pass")
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    a, kind = _Args("score_passes"), _wkind(w_dtype)
    hs, ls, ts = (ctypes.c_void_p * max(n, 1))(), (ctypes.c_void_p * max(n, 1))(), (ctypes.c_void_p * max(n, 1))()
    for b, p in enumerate(arr.tolist()):
        T, M, G, _ = plan._sizes(p)
        hs[b] = a(hidden[b], f"hidden[{b}]", "bf16", (M if slot_rows else T) * d_model)
        ls[b] = a(row_lse[b], f"row_lse[{b}]", "f32", M)
        ts[b] = a(token_lp[b], f"token_lp[{b}]", "f32", G)
    _check(lib().spinf_score_passes(plan.handle, n, ptr, hs, HIDDEN_SLOT_ROWS if slot_rows else HIDDEN_PASS_ROWS,
                                    a(w, "w", kind, vocab * d_model),
                                    a(w_scale, "w_scale", "f32", vocab), w_dtype, d_model, vocab, ls, ts,
                                    a(workspace, "workspace", "bytes"), int(workspace_bytes), _stream(stream)))


def score_static(plan, p, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp, stream=None):
    """``spinf_score_static``: scoring with the library's own fixed device scratch (no allocation)."""
    args = _score_args(_Args("score_static"), plan, p, hidden, w, w_scale, w_dtype, d_model, vocab, row_lse, token_lp)
    _check(lib().spinf_score_static(plan.handle, p, *args, _stream(stream)))


def decode_attention(plan, p, q, k_pass, v_pass, k_dec, v_dec, anchor, parent, q_row, o, n_q_heads, n_kv_heads,
                     d_head, scale=0.0, stream=None):
    """One decoding step of searched slots (spinf_decode_attention); anchor, parent, q_row are
    device int32 tensors."""
    a = _Args("decode_attention")
    T = plan._sizes(p)[0]
    n_dec, n_q = anchor.numel(), q_row.numel()
    nq, nkv, ndec = n_q * n_q_heads * d_head, T * n_kv_heads * d_head, n_dec * n_kv_heads * d_head
    _check(lib().spinf_decode_attention(plan.handle, p, a(q, "q", "bf16", nq), a(k_pass, "k_pass", "bf16", nkv),
                                        a(v_pass, "v_pass", "bf16", nkv), a(k_dec, "k_dec", "bf16", ndec),
                                        a(v_dec, "v_dec", "bf16", ndec), n_dec, a(anchor, "anchor", "i32", n_dec),
                                        a(parent, "parent", "i32", n_dec), a(q_row, "q_row", "i32", n_q), n_q,
                                        a(o, "o", "bf16", nq), n_q_heads, n_kv_heads, d_head, float(scale),
                                        _stream(stream)))


def score_rows(plan, hidden, w, w_scale, w_dtype, d_model, vocab, k, row_lse, top_tok, top_lp, token_set=None,
               token_sets=None, workspace=None, stream=None):
    """Next-token answers at caller-given rows (spinf_score_rows); token_set: a device int32 tensor or None."""
    import torch
    a, kind = _Args("score_rows"), _wkind(w_dtype)
    n = hidden.shape[0]
    n_sets = 0 if token_sets is None else int(token_sets.shape[0])
    args = (a(hidden, "hidden", "bf16", n * d_model), n, a(w, "w", kind, vocab * d_model),
            a(w_scale, "w_scale", "f32", vocab), w_dtype, d_model, vocab, a(token_set, "token_set", "i32", n),
            a(token_sets, "token_sets", "words", n_sets * (-(-vocab // 32))), n_sets, k,
            a(row_lse, "row_lse", "f32", n), a(top_tok, "top_tok", "i32", n * k), a(top_lp, "top_lp", "f32", n * k))
    if workspace is None:
        workspace = torch.empty(max(1, lib().spinf_score_rows_workspace_bytes(n, vocab, d_model, w_dtype, k)),
                                dtype=torch.uint8, device=hidden.device)
    _check(lib().spinf_score_rows(plan.handle, *args, a(workspace, "workspace", "bytes"),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))
