"""The C-ABI library builds, loads and exports what include/ss_scan.h declares
(CPU only: no compute call is made without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ss_scan.h")


@pytest.fixture(scope="module")
def built():
    from selective_state_space_136_b300 import build
    return build.build()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(built):
    lib = ctypes.CDLL(built["libss_scan.so"])
    names = _declared_functions()
    assert {"ss_create", "ss_destroy", "ss_scan_fwd", "ss_state_update"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layout_matches_binding(built, tmp_path):
    """ctypes mirrors of the argument structs have the C layout."""
    import selective_state_space_136_b300 as ss
    structs = {"ss_scan_args": ss.ScanArgs, "ss_update_args": ss.UpdateArgs,
               "ss_scan_bwd_args": ss.ScanBwdArgs, "ss_ssd_args": ss.SsdArgs,
               "ss_conv1d_args": ss.Conv1dArgs, "ss_conv1d_update_args": ss.Conv1dUpdateArgs,
               "ss_conv_scan_args": ss.ConvScanArgs}
    prog = tmp_path / "layout.c"
    body = ['#include <stdio.h>', '#include <stddef.h>', '#include "ss_scan.h"', "int main(void){"]
    for cname, cls in structs.items():
        body.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for f, _ in cls._fields_:
            body.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, f, cname, f))
    body.append("return 0;}")
    prog.write_text("\n".join(body))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(prog)])
    seen = set()
    for line in subprocess.check_output([str(exe)]).decode().split("\n"):
        if not line:
            continue
        cname, name, val = line.split()
        cls = structs[cname]
        if name == "size":
            assert int(val) == ctypes.sizeof(cls), cname
        else:
            assert getattr(cls, name).offset == int(val), (cname, name)
        seen.add(cname)
    assert seen == set(structs)


def test_enum_constants_match_binding(tmp_path):
    """Every enumerator the header defines has the same value in the binding."""
    import selective_state_space_136_b300 as ss
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(SS_[A-Z0-9_]+)\s*=", text)))
    assert {"SS_OK", "SS_OPT_SSD_PATH", "SS_SSD_PATH_TCGEN05", "SS_DISC_ZOH"} <= set(names)
    prog = tmp_path / "enums.c"
    prog.write_text("\n".join(['#include <stdio.h>', '#include "ss_scan.h"', "int main(void){"] +
                              ['printf("%s %%d\\n", (int)%s);' % (n, n) for n in names] +
                              ["return 0;}"]))
    exe = tmp_path / "enums"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(prog)])
    for line in subprocess.check_output([str(exe)]).decode().split("\n"):
        if line:
            name, val = line.split()
            assert getattr(ss, name) == int(val), name


def test_host_validation_without_gpu(built):
    import selective_state_space_136_b300 as ss
    L = ss.lib()
    assert L.ss_scan_fwd(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_state_update(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_conv1d_fwd(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_scan_bwd(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_ssd_fwd(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_conv1d_update(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_scan_fwd_noalloc(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_conv_scan_fwd(None, None, None) == ss.SS_ERR_INVALID_ARG
    assert L.ss_set_option(None, 0, 0) == ss.SS_ERR_INVALID_ARG
    assert L.ss_destroy(None) == ss.SS_OK
    assert ss.status_string(ss.SS_ERR_TIMEOUT) == "device wait timed out"
    assert ss.status_string(99) == "unknown status"


def test_create_fails_cleanly_without_gpu(built):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import selective_state_space_136_b300 as ss
    h = ctypes.c_void_p()
    assert ss.lib().ss_create(ctypes.byref(h), 0) == ss.SS_ERR_CUDA
    assert not h.value


def test_binding_refuses_cpu_tensors(built):
    import torch
    import selective_state_space_136_b300 as ss
    x = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        ss.ss_scan_fwd(x, x, torch.zeros(4, 4), torch.zeros(1, 4, 8), torch.zeros(1, 4, 8))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import selective_state_space_136_b300 as ss
    monkeypatch.setattr(ss, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(ss, "_lib", None)
    with pytest.raises(RuntimeError):
        ss.lib()
