"""CPU dry run of bench.py (TEST INFRASTRUCTURE ONLY): CUDA streams and events faked,
"device" tensors on the CPU, the library's device entry points stubbed to OK (the planner,
schedules, sizes and collect are real), and the binding's dtype / contiguity / size checks
kept with only its CUDA-placement check relaxed.  Kernel results are not computed, so the
figures printed are meaningless; what is checked is that every leg of the benchmark runs
and prints its line.  Usage: python tests/bench_dry_run.py [bench arguments]."""
import contextlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import torch  # noqa: E402

class FakeEvent:
    def __init__(self, *a, **k): pass
    def record(self, *a, **k): pass
    def elapsed_time(self, other): return 1.0
    def synchronize(self): pass
    def query(self): return True
class FakeStream:
    cuda_stream = 0
    def __init__(self, *a, **k): pass
    def synchronize(self): pass
    def wait_event(self, e): pass
    def wait_stream(self, s): pass
torch.cuda.Event = FakeEvent
torch.cuda.Stream = FakeStream
torch.cuda.stream = lambda s=None: contextlib.nullcontext()
torch.cuda.synchronize = lambda *a, **k: None
torch.cuda.set_device = lambda *a, **k: None
torch.cuda.current_device = lambda: 0
torch.cuda.current_stream = lambda *a, **k: FakeStream()
torch.cuda.is_available = lambda: True
torch.cuda.device_count = lambda: 1

def _cpu(d):
    if d is None: return None
    dd = d if isinstance(d, torch.device) else torch.device(d)
    return torch.device('cpu') if dd.type == 'cuda' else dd
for name in ('empty', 'zeros', 'ones', 'full', 'randn', 'rand', 'arange', 'empty_like', 'full_like', 'zeros_like',
             'as_tensor', 'tensor', 'randint'):
    orig = getattr(torch, name)
    def wrap(*a, _orig=orig, **k):
        if 'device' in k: k['device'] = _cpu(k['device'])
        k.pop('pin_memory', None)
        return _orig(*a, **k)
    setattr(torch, name, wrap)
# the stubbed kernels write nothing: buffers start as zeros, so the results read back are finite
_empty, _empty_like = torch.empty, torch.empty_like
torch.empty = lambda *a, **k: _empty(*a, **k).zero_()
torch.empty_like = lambda *a, **k: _empty_like(*a, **k).zero_()
_Gen = torch.Generator
torch.Generator = lambda device=None: _Gen(device='cpu')
_to = torch.Tensor.to
def to(self, *a, **k):
    a = list(a)
    if a and isinstance(a[0], (str, torch.device)) and torch.device(a[0]).type == 'cuda': a[0] = 'cpu'
    if 'device' in k: k['device'] = _cpu(k['device'])
    return _to(self, *a, **k)
torch.Tensor.to = to
torch.Tensor.cuda = lambda self, *a, **k: self
torch.Tensor.pin_memory = lambda self, *a, **k: self
_copy = torch.Tensor.copy_
torch.Tensor.copy_ = lambda self, src, non_blocking=False: _copy(self, src)

import branch_packed_scoring_gb300 as spinf  # noqa: E402
real = spinf.lib()
DEVICE = {"spinf_plan_upload", "spinf_plan_upload_to", "spinf_plan_upload_pinned", "spinf_branch_attention", "spinf_score", "spinf_score_extract",
          "spinf_score_passes",
          "spinf_score_static", "spinf_device_status", "spinf_device_selftest", "spinf_rope_tree", "spinf_linear",
          "spinf_qkv_rope", "spinf_quantize_static", "spinf_decode_attention", "spinf_score_rows"}
calls = {}
class Proxy:
    def __getattr__(self, n):
        if n in DEVICE:
            def f(*a):
                calls[n] = calls.get(n, 0) + 1
                return 0
            return f
        return getattr(real, n)
spinf._lib = Proxy()
def check(self, x, what, kind, n=None):
    if x is None or isinstance(x, int): return x
    if not hasattr(x, 'is_cuda'): self.bad(f"{what} must be a torch tensor or a device address")
    dts = spinf._kinds()[kind]
    if dts is not None and x.dtype not in dts: self.bad(f"{what} has dtype {x.dtype}; {kind} expected")
    if not x.is_contiguous(): self.bad(f"{what} must be contiguous")
    if n is not None and x.numel() < n: self.bad(f"{what} holds {x.numel()} elements; the call needs {n}")
    return x.data_ptr()
spinf._Args.__call__ = check

import bench  # noqa: E402
sys.argv = ['bench.py'] + sys.argv[1:]
bench.main()
print("device calls:", calls, file=sys.stderr)
