"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (CPU only; no compute calls)."""
import ctypes
import os
import re

import pytest

from hyper_connection_rank_gb300 import _binding as B
from hyper_connection_rank_gb300 import build as gpu_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gpu_build.build()
    return B.load_library()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(hc_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "hc_lowrank_mix" in names and len(names) >= 7
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(B.EXPORTS) <= set(names)


def test_library_is_built_for_sm103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(gpu_build.NVCC_FLAGS)
    assert "--use_fast_math" not in gpu_build.NVCC_FLAGS


def test_defaults_and_status_strings(L):
    a = L.hc_attrs_default()
    assert (a.epsilon, a.reduction_scale, a.silu_alpha, a.gate_div, a.gate_mul, a.flags) == \
        (ctypes.c_float(1e-5).value, 1.0, 1.0, 1.0, 1.0, 0)
    assert L.hc_status_string(0) == b"HC_OK"
    assert L.hc_status_string(3) == b"HC_ERR_WORKSPACE"


FAKE = {n: 0x100000 * (i + 1) for i, n in enumerate(
    ["streams", "norm_scale", "down_w", "up_w", "inject_w", "prev_out", "prev_gate", "pre", "post", "sout", "ws"])}


def call(**over):
    a = dict(FAKE, rows=2, C=4, H=64, R=16, dt=B.HC_BF16, ws_bytes=1 << 16)
    a.update(over)
    attrs = B.make_attrs()
    return B.raw_call(a["streams"], a["norm_scale"], a["down_w"], a["up_w"], a["inject_w"], a["prev_out"],
                      a["prev_gate"], a["rows"], a["C"], a["H"], a["R"], attrs, a["dt"], a["pre"], a["post"],
                      a["sout"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("over", [
    dict(rows=-1), dict(C=0), dict(H=0), dict(R=0), dict(dt=7),
    dict(down_w=None), dict(norm_scale=None), dict(up_w=None), dict(inject_w=None),
    dict(prev_gate=None), dict(prev_out=None),
    dict(streams=None), dict(pre=None), dict(post=None),
    dict(pre=FAKE["streams"] + 64),            # output inside an input
    dict(sout=FAKE["streams"]),                 # streams_out aliasing streams
    dict(post=FAKE["pre"] + 2),                 # two outputs overlapping
    dict(ws=FAKE["down_w"]),                    # workspace over a weight
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_rejected_before_launch(L, over):
    assert call(**over) == B.HC_ERR_INVALID_ARG
    assert len(L.hc_last_error()) > 0


def test_zero_rows_is_ok_without_row_pointers(L):
    assert call(rows=0, streams=None, pre=None, post=None, sout=None, prev_out=None, prev_gate=None) == B.HC_OK


def test_no_gpu_fails_loudly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() in (B.HC_ERR_CUDA, B.HC_ERR_UNSUPPORTED)


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "hc_lowrank_mix.h"
#include "hc_row_ops.h"

int main(void) {
  hc_attrs_t a = hc_attrs_default();
  char fake[64];
  hc_status_t s;
  if (a.silu_alpha != 1.0f || a.flags != 0u) return 1;
  if (strcmp(hc_status_string(HC_ERR_WORKSPACE), "HC_ERR_WORKSPACE") != 0) return 2;
  /* invalid sizes are refused on the host, before any device access */
  s = hc_lowrank_mix(fake, fake, fake, fake, fake, NULL, NULL, -1, 4, 64, 16, &a, HC_BF16,
                     fake, fake, NULL, NULL, 0, NULL);
  if (s != HC_ERR_INVALID_ARG || hc_last_error()[0] == '\0') return 3;
  /* zero rows launch nothing and need no row pointers */
  s = hc_lowrank_mix(NULL, fake, fake, fake, fake, NULL, NULL, 0, 4, 64, 16, NULL, HC_F32,
                     NULL, NULL, NULL, NULL, 0, NULL);
  if (s != HC_OK) return 4;
  if (hc_inv_rms(fake, 1, 0, 1e-6f, HC_F32, (float*)fake, NULL) != HC_ERR_INVALID_ARG) return 5;
  if (hc_engram_gate(fake, fake, fake, fake, fake, 0, 4, 64, 1e-5f, HC_F16, fake, NULL) != HC_OK) return 6;
  printf("ok %s\n", hc_status_string(HC_OK));
  return 0;
}
"""


def test_headers_serve_a_plain_c_program(L, tmp_path):
    """include/*.h compile as strict C99 (no C++ or CUDA types in the
    signatures), and a C program linked against the library gets the
    documented host-side results (argument errors, zero rows) without a GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    lib_dir = os.path.dirname(B.LIB_PATH)
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), B.LIB_PATH, f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok HC_OK", (r.returncode, r.stdout, r.stderr)
