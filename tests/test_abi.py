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
