"""The C-ABI library loads without a GPU and exports every symbol the header declares."""
import re
import os

import pytest

from conftest import ROOT


def _declared():
    text = open(os.path.join(ROOT, "include", "spinf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spinf_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree(spinf):
    assert _declared() == sorted(spinf.SYMBOLS)


def test_every_declared_symbol_is_exported(spinf):
    L = spinf.lib()
    for name in _declared():
        assert hasattr(L, name), name


def test_fingerprint_and_status_strings(spinf):
    fp = spinf.fingerprint()
    assert "sm_103a" in fp and "tcgen05" in fp
    L = spinf.lib()
    names = [L.spinf_status_string(s).decode() for s in range(8)]
    assert names[0] == "ok" and len(set(names)) == 8


def test_device_calls_fail_loudly_without_upload(spinf):
    plan = spinf.Plan([([1, 2, 3], [([4, 5], [[6], [7]])])])
    with pytest.raises(spinf.SpinfError) as e:
        spinf.branch_attention(plan, 0, 16, 16, 16, 16, 4, 2, 64, stream=0)
    assert e.value.status_name == "INVALID"
    with pytest.raises(spinf.SpinfError):
        spinf.score(plan, 0, 16, 16, None, 0, 256, 1024, 16, 16, 16, 1 << 20, stream=0)


def test_upload_to_validates_before_any_device_work(spinf):
    """Caller-owned descriptor memory: size and alignment are checked first (no GPU needed)."""
    L = spinf.lib()
    plan = spinf.Plan([([1, 2, 3], [([4, 5], [[6], [7]])])])
    need = plan.descriptor_bytes(0)
    info = plan.pass_info(0)
    assert need >= 256 + 4 * (2 * info.T_pad + 8 * info.T_pad)   # end, pos, row runs and the error word
    assert plan.descriptor_bytes(5) == 0
    for ptr, size in ((None, need), (4096 + 16, need), (4096, need - 1)):
        st = L.spinf_plan_upload_to(plan.handle, 0, ptr, size, None)
        assert spinf.STATUS_NAMES[st] == "INVALID"
    assert spinf.STATUS_NAMES[L.spinf_plan_upload_to(plan.handle, 3, 4096, need, None)] == "INVALID"
    # the pinned-staging variant refuses a NULL staging buffer first
    assert spinf.STATUS_NAMES[L.spinf_plan_upload_pinned(plan.handle, 0, 4096, need, None, need, None)] == "INVALID"


def test_selftest_needs_an_uploaded_plan(spinf):
    """No device work happens for a plan without an error word (no GPU needed)."""
    plan = spinf.Plan([([1, 2, 3], [([4, 5], [[6], [7]])])])
    st = spinf.lib().spinf_device_selftest(plan.handle, 30, None)
    assert spinf.STATUS_NAMES[st] == "INVALID"


def test_layer_and_decode_calls_validate_before_any_device_work(spinf):
    """Arguments of the projection, decode and row-scoring calls are checked on the host first
    (no GPU needed): a plan that was never uploaded has no error word, bad sizes are refused."""
    L = spinf.lib()
    plan = spinf.Plan([([1, 2, 3], [([4, 5], [[6], [7]])])])
    names = spinf.STATUS_NAMES
    # spinf_linear needs an uploaded plan (its device error word)
    assert names[L.spinf_linear(plan.handle, 4096, 4096, None, 1.0, 0, 4096, 8, 64, 64, None)] == "INVALID"
    assert names[L.spinf_qkv_rope(plan.handle, 0, 4096, 4096, None, 1.0, 0, 256, 4, 2, 64, 10000.0, 4096, 4096,
                                  4096, None)] == "INVALID"
    assert names[L.spinf_decode_attention(plan.handle, 0, 4096, 4096, 4096, 4096, 4096, 1, 4096, 4096, 4096, 1,
                                          4096, 4, 2, 64, 0.0, None)] == "INVALID"
    assert names[L.spinf_score_rows(plan.handle, 4096, 1, 4096, None, 0, 256, 1024, None, None, 0, 8, 4096, 4096,
                                    4096, 4096, 1 << 20, None)] == "INVALID"
    assert names[L.spinf_quantize_static(4096, 0.0, 4096, 8, None)] == "INVALID"     # scale must be positive
    assert names[L.spinf_quantize_static(4096, 1.0, 4096, 7, None)] == "INVALID"     # n a multiple of 8
    assert L.spinf_score_rows_workspace_bytes(0, 1024, 256, 0, 8) == 0
    assert L.spinf_score_rows_workspace_bytes(4, 1024, 256, 0, 17) == 0
    assert L.spinf_score_rows_workspace_bytes(4, 1024, 256, 0, 8) > 4 * 256 * 2


def test_binding_checks_tensors_before_the_call(spinf):
    """The binding refuses a tensor of the wrong dtype, a strided view, a buffer smaller than
    the call reads or writes, and a host tensor, before anything reaches the library (no GPU
    needed).  Raw addresses (ints) pass through unchecked, so each case below gives them for
    the arguments ahead of the one under test."""
    torch = pytest.importorskip("torch")
    plan = spinf.Plan([([1, 2, 3], [([4, 5], [[6], [7]])])], vocab=1024)
    info = plan.pass_info(0)
    T, M, G = info.T_pad, info.M, info.G
    A = 4096
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)  # noqa: E731
    f32 = lambda n: torch.zeros(n)  # noqa: E731
    i32 = lambda n: torch.zeros(n, dtype=torch.int32)  # noqa: E731
    q, kv, w = bf(T, 4, 64), bf(T, 2, 64), bf(1024, 256)
    ws = torch.zeros(16, dtype=torch.uint8)
    cases = [
        (lambda: spinf.branch_attention(plan, 0, q.float(), A, A, A, 4, 2, 64), "q has dtype torch.float32"),
        (lambda: spinf.branch_attention(plan, 0, A, A, A, q.transpose(0, 1), 4, 2, 64), "o must be contiguous"),
        (lambda: spinf.branch_attention(plan, 0, A, kv[:T - 1], A, A, 4, 2, 64), "k holds"),
        (lambda: spinf.branch_attention(plan, 0, q, A, A, A, 4, 2, 64), "q must be a CUDA tensor"),
        (lambda: spinf.branch_attention(plan, 0, [1], A, A, A, 4, 2, 64), "q must be a torch tensor"),
        (lambda: spinf.score(plan, 0, A, A, None, spinf.DTYPE_BF16, 256, 1024, f32(M - 1), A, A,
                             workspace_bytes=1 << 20), "row_lse holds"),
        (lambda: spinf.score(plan, 0, A, w, None, spinf.DTYPE_E4M3, 256, 1024, A, A, ws), "w has dtype"),
        (lambda: spinf.score(plan, 0, A, A, None, spinf.DTYPE_BF16, 256, 1024, A, A, A, workspace_bytes=1 << 20,
                             extract={"top_tok": f32(8), "top_lp": A}), "top_tok has dtype"),
        (lambda: spinf.score_static(plan, 0, bf(1, 256), A, None, spinf.DTYPE_BF16, 256, 1024, A, A),
         "hidden holds"),
        (lambda: spinf.rope_tree(plan, 0, A, kv[:1], 4, 2, 64), "k holds"),
        (lambda: spinf.linear(plan, f32(512).view(8, 64), bf(32, 64), A), "x has dtype"),
        (lambda: spinf.qkv_rope(plan, 0, bf(T, 256), A, A, A, A, 4, 2, 64, w_scale=f32(10),
                                w_dtype=spinf.DTYPE_E4M3), "x has dtype"),
        (lambda: spinf.quantize_static(f32(64), 0.5, A), "x has dtype"),
        (lambda: spinf.decode_attention(plan, 0, A, A, A, A, A, torch.zeros(3, dtype=torch.int64), A, i32(2), A,
                                        4, 2, 64), "anchor has dtype"),
        (lambda: spinf.score_rows(plan, bf(4, 256), w, None, spinf.DTYPE_BF16, 256, 1024, 8, A, A, f32(31),
                                  workspace=ws), "hidden must be a CUDA tensor"),
    ]
    for fn, words in cases:
        with pytest.raises(spinf.SpinfError) as e:
            fn()
        assert e.value.status_name == "INVALID" and words in str(e.value), str(e.value)


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_is_plain_c_and_cpp(lang, std):
    """The public header compiles on its own as strict C99 (no C++ or CUDA types leak into
    the ABI) and as C++17."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "spinf.h")
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", "-x", lang,
                        header], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_caller(spinf, tmp_path):
    """A C program plans and collects through the library alone (host calls, no Python in
    between); the layout and the results are the hand-derived ones: content 4 rows, template
    2, trie node 1, floor 3 (10 rows, 4 scoring rows, 6 gathered tokens); token probabilities
    1/2 for [7] and 1/4 * 1/2 for [8, 9] give p = 0.8 / 0.2 and residual 0.375; the floor's
    1/2 and 1/2 * 1/2 give 2/3 / 1/3 and residual 0.25."""
    import shutil
    import subprocess
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no host compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    lib_dir = os.path.dirname(spinf.LIB_PATH)
    exe = str(tmp_path / "c_client")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(here, "c_client.c"), "-o", exe, "-L", lib_dir, "-lspinf",
                        f"-Wl,-rpath,{lib_dir}", "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    first, second = out.stdout.splitlines()
    v = first.split()
    assert [int(x) for x in v[:6]] == [1, 10, 4, 6, 1, 2]
    got = [float(x) for x in v[6:]]
    want = [0.8, 0.2, 0.375, 2 / 3, 1 / 3, 0.25]
    assert all(abs(a - b) < 1e-6 for a, b in zip(got, want)), got
    # searched slot: one slot, k = 2, its answer returned as set; no residual for it
    v = second.split()
    assert [int(x) for x in v[:5]] == [1, 2, 1, 42, 17]
    assert [float(x) for x in v[5:7]] == [-0.5, -1.5] and v[7] == "1"
    assert all(abs(float(x) - 0.375) < 1e-6 for x in v[8:10])


def test_score_passes_rejects_bad_lists(spinf):
    """spinf_score_passes checks its pass list before touching the device: a pass listed twice
    or out of range is INVALID, more than SPINF_SCORE_MAX_PASSES passes is LIMIT; the workspace
    query returns 0 for such lists."""
    from synth import workloads as wl
    plan = spinf.Plan(wl.stress(n_questions=40, content_tokens=100, vocab=1000), vocab=1000, token_budget=512)
    n = plan.num_passes
    assert n >= 3
    for passes, status in (([0, 0], "INVALID"), ([n], "INVALID"), ([-1], "INVALID"), (list(range(n)) * 12, "LIMIT")):
        assert spinf.score_passes_workspace_bytes(plan, passes, 1000, 512) == 0
        k = len(passes)
        with pytest.raises(spinf.SpinfError) as e:
            spinf.score_passes(plan, passes, [0] * k, 0, None, spinf.DTYPE_BF16, 512, 1000, [0] * k, [0] * k, 0, 0,
                               stream=0)
        assert e.value.status_name == status, passes
    assert spinf.score_passes_workspace_bytes(plan, [0, 1], 1000, 512) > 0
