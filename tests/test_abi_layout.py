"""The Python mirrors of the C ABI's structs (the packed sampler settings,
the logit-bias entries and the GEMM fusion options) have the layout kinv.h
gives them: every field's offset and the struct's size, as a C compiler lays
them out.  No GPU needed."""
import ctypes
import os
import shutil
import subprocess

import pytest

from invariant_deterministic_gb300 import kinv, synth

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))

STRUCTS = {
    "kinv_sampling_params": [f for f in synth.SAMPLING_DTYPE.names],
    "kinv_logit_bias": [f for f in synth.BIAS_DTYPE.names],
    "kinv_gemm_fusion": [f for f, _ in kinv.GemmFusion._fields_],
}


def _c_layout(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kinv.h"', "int main(void) {"]
    for s, fields in STRUCTS.items():
        lines.append(f'  printf("{s} size %zu\\n", sizeof({s}));')
        for f in fields:
            lines.append(f'  printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines.append("  return 0;\n}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    layout = {}
    for line in out.splitlines():
        s, f, v = line.split()
        layout[(s, f)] = int(v)
    return layout


def test_struct_layouts_match_the_header(tmp_path):
    c = _c_layout(tmp_path)
    for dt, name in ((synth.SAMPLING_DTYPE, "kinv_sampling_params"), (synth.BIAS_DTYPE, "kinv_logit_bias")):
        assert dt.itemsize == c[(name, "size")], name
        for f in dt.names:
            assert dt.fields[f][1] == c[(name, f)], (name, f)
    assert ctypes.sizeof(kinv.GemmFusion) == c[("kinv_gemm_fusion", "size")]
    for f, _ in kinv.GemmFusion._fields_:
        assert getattr(kinv.GemmFusion, f).offset == c[("kinv_gemm_fusion", f)], f


def test_sampling_struct_packing():
    """Row i's logit_bias points at its first entry of bias_entries(), its
    count and every other setting land in their fields; a bias list needs a
    device base address."""
    P = kinv.SamplingParams
    rows = [P(seed=1), P(seed=2, logit_bias={5: 1.5, 9: -2.0}, typical_p=0.5),
            P(seed=3, presence_penalty=0.25, frequency_penalty=0.5), P(seed=4, logit_bias={7: 3.0})]
    entries, starts = synth.bias_entries(rows)
    assert starts == [0, 0, 2, 2]
    assert entries.tolist() == [(5, 1.5), (9, -2.0), (7, 3.0)]
    a = synth.sampling_struct(rows, bias_base=0x10000)
    assert a["logit_bias"].tolist() == [0, 0x10000, 0, 0x10000 + 2 * synth.BIAS_DTYPE.itemsize]
    assert a["n_logit_bias"].tolist() == [0, 2, 0, 1]
    assert a["seed"].tolist() == [1, 2, 3, 4]
    assert a["typical_p"].tolist() == [1.0, 0.5, 1.0, 1.0]
    assert a["presence_penalty"].tolist()[2] == 0.25 and a["frequency_penalty"].tolist()[2] == 0.5
    with pytest.raises(ValueError):
        synth.sampling_struct(rows)
