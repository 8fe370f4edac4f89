"""CPU checks of the C-ABI library: it builds, loads without a GPU, and
exports every function include/pa.h declares. No compute calls."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pa_create", "pa_destroy", "pa_load_library", "pa_load_netlist", "pa_load_events", "pa_run",
              "pa_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import gate_level_power_gb300 as glp
    glp.build()
    lib = ctypes.CDLL(glp.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(glp.EXPORTS) == set(declared_functions())


def test_version_and_defaults_without_gpu():
    import gate_level_power_gb300 as glp
    glp.build()
    assert glp.pa_version() == 3
    p = glp.pa_default_params()
    assert p.n_cycles == 1 and abs(p.vdd - 0.9) < 1e-12 and p.t_clk_ns == 1.0


def test_binding_struct_layouts_match_header(tmp_path):
    # every field offset and struct size as the C compiler lays out pa.h
    import subprocess

    import gate_level_power_gb300 as glp
    structs = {"pa_library": glp.PaLibrary, "pa_netlist": glp.PaNetlist, "pa_events": glp.PaEvents,
               "pa_run_params": glp.PaRunParams, "pa_result": glp.PaResult}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "pa.h"', 'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            cf = {"waveform": "waveform_w"}.get(fname, fname)
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {cf}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe)])
    got = {}
    for line in subprocess.check_output([str(exe)]).decode().split("\n"):
        if line:
            a, b, c = line.split()
            got[(a, b)] = int(c)
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)


def test_create_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import gate_level_power_gb300 as glp
    with pytest.raises(glp.PaError) as ei:
        glp.pa_create(0)
    assert ei.value.code == glp.PA_ERR_CUDA


def test_ctypes_structs_match_the_c_layout(tmp_path):
    # the binding's ctypes mirrors of the header's structs: sizes and offsets
    import subprocess
    import gate_level_power_gb300 as glp
    structs = {"pa_run_params": glp.PaRunParams, "pa_result": glp.PaResult, "pa_events": glp.PaEvents}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "pa.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
        for f in cls._fields_:
            lines.append(f'  printf("{cname}.{f[0]} %zu\\n", offsetof({cname}, {f[0]}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe)])
    got = dict(line.split() for line in subprocess.check_output([str(exe)]).decode().splitlines())
    for cname, cls in structs.items():
        assert int(got[cname]) == ctypes.sizeof(cls), cname
        for f in cls._fields_:
            assert int(got[f"{cname}.{f[0]}"]) == getattr(cls, f[0]).offset, (cname, f[0])
