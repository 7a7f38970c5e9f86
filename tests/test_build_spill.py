"""The build refuses register spills ("deepseek-ai/FlashMLA", "Key technical
details": the kernels are built with a register-spill check).  The ptxas
report of every translation unit is parsed; any kernel with nonzero spill
stores or loads stops the build before the library is linked.  These tests
feed the parser and build() synthetic ptxas reports (no nvcc, no GPU)."""
import os

import pytest

from fp4_kv_cache_sparse_gb300 import build as B

KERNEL = "_ZN3mla12_GLOBAL__N_120sparse_decode_kernelILi64EEEvNS_12DecodeParamsE14CUtensorMap_st"


def _report(kernel, stores, loads, stack=0):
    return (f"ptxas info    : 0 bytes gmem\n"
            f"ptxas info    : Compiling entry function '{kernel}' for 'sm_103a'\n"
            f"ptxas info    : Function properties for {kernel}\n"
            f"    {stack} bytes stack frame, {stores} bytes spill stores, {loads} bytes spill loads\n"
            f"ptxas info    : Used 168 registers, used 1 barriers\n")


def test_clean_report_passes():
    B.refuse_spills(["decode.cu"], [_report(KERNEL, 0, 0)])
    assert B._check_spills("decode.cu", _report(KERNEL, 0, 0)) == []


@pytest.mark.parametrize("stores,loads", [(8, 8), (8, 0), (0, 4)])
def test_spilling_kernel_is_refused_by_name(stores, loads):
    logs = [_report("_Z9other_kernv", 0, 0), _report(KERNEL, stores, loads, stack=8)]
    with pytest.raises(B.SpillError) as e:
        B.refuse_spills(["combine.cu", "decode.cu"], logs)
    msg = str(e.value)
    assert KERNEL in msg and "decode.cu" in msg
    assert "_Z9other_kernv" not in msg


def test_device_function_report_is_attributed():
    # ptxas reports non-inlined device functions as "Function properties for"
    # without a "Compiling entry function" line.
    log = ("ptxas info    : Function properties for _ZN3mla6helperEv\n"
           "    16 bytes stack frame, 16 bytes spill stores, 16 bytes spill loads\n")
    bad = B._check_spills("api.cu", log)
    assert len(bad) == 1 and "_ZN3mla6helperEv" in bad[0]


def test_build_stops_before_linking(tmp_path, monkeypatch):
    """build() itself raises on a spilling report and leaves no library."""
    monkeypatch.setattr(B, "BUILD", str(tmp_path))
    monkeypatch.setattr(B, "LIB", str(tmp_path / "libmla.so"))
    monkeypatch.setattr(B, "SOURCES", ["a.cu", "b.cu"])
    logs = {"a.cu": _report("_Z1av", 0, 0), "b.cu": _report(KERNEL, 24, 24, stack=24)}
    monkeypatch.setattr(B, "_compile", lambda src: (str(tmp_path / (src + ".o")), logs[src]))

    def no_link(*a, **k):
        raise AssertionError("the library must not be linked")

    monkeypatch.setattr(B.subprocess, "run", no_link)
    with pytest.raises(B.SpillError):
        B.build(force=True)
    assert not os.path.exists(tmp_path / "libmla.so")
    assert "24 bytes spill stores" in open(tmp_path / "ptxas.log").read()
