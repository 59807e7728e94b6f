"""The C-ABI library builds, loads and exports what include/libattn.h declares.

Runs without a GPU: only argument checks that return before any device work
are exercised, plus the loud failure when no sm_103 device is present.
"""
import ctypes as C
import os
import re

import pytest
import torch

from exact_attention_73_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "libattn.h")


def declared():
    txt = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", txt)


def test_header_declares_the_binding_exports():
    assert sorted(declared()) == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert binding.attn_version().startswith("libattn")
    for code, name in binding.STATUS.items():
        assert binding.attn_status_string(code).startswith(name)


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, Hq=2, Hkv=1, N=8, d=64, dt=0):
    P = lambda x: C.c_void_p(x) if x else None
    return lib.attn_fwd(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, N, d, 0.125, 0, dt, None)


def test_argument_checks_before_any_device_work(lib):
    assert _fwd(lib, q=0) == 1                      # NULL
    assert _fwd(lib, k=0x1008) == 2                 # not 16-byte aligned
    assert _fwd(lib, N=0) == 3                      # shape
    assert _fwd(lib, B=0) == 3
    assert _fwd(lib, d=96) == 4                     # head dim
    assert _fwd(lib, Hq=3, Hkv=2) == 5              # GQA
    assert _fwd(lib, dt=2) == 6                     # E4M3 goes through attn_fwd_fp8
    P = C.c_void_p
    # varlen: nseq, T and max_seqlen are checked
    assert lib.attn_fwd_varlen(P(16), P(16), P(16), P(16), P(16), P(16), 0, 10, 5, 2, 1, 64, 0.1, 0, 0, None) == 3
    assert lib.attn_fwd_varlen(P(16), P(16), P(16), P(16), P(16), P(16), 2, 10, 11, 2, 1, 64, 0.1, 0, 0, None) == 3
    assert lib.attn_fwd_varlen(P(16), P(16), P(16), P(16), P(16), None, 2, 10, 5, 2, 1, 64, 0.1, 0, 0, None) == 1
    # FP8 forward blocking: keys per KV tile by head dimension (no device work)
    assert [binding.attn_fwd_fp8_kv_tile(d) for d in (64, 128, 256, 100)] == [128, 128, 128, 0]
    # decode: splits within [1, ceil(Nmax/128)], group size <= 128, workspace
    wdec = binding.attn_decode_fp8_workspace_size(2, 8, 128, 3)
    assert wdec == (3 * 2 * 8 * 128 * 4 + 255) // 256 * 256 + 256
    dargs = [P(16)] * 6 + [None, P(16), P(16), P(16)]
    assert lib.attn_decode_fp8(*dargs, wdec, 2, 8, 2, 300, 128, 0.1, 4, None) == 3            # > ceil(300/128) splits
    assert lib.attn_decode_fp8(*dargs, wdec, 2, 8, 2, 300, 128, 0.1, 0, None) == 3
    assert lib.attn_decode_fp8(*dargs, wdec - 1, 2, 8, 2, 300, 128, 0.1, 3, None) == 7
    assert lib.attn_decode_fp8(*dargs, wdec, 2, 8, 3, 300, 128, 0.1, 3, None) == 5
    assert lib.attn_decode_fp8(*dargs, wdec, 2, 8, 2, 300, 96, 0.1, 3, None) == 4
    assert lib.attn_decode_fp8(*dargs, wdec, 1, 256, 1, 300, 128, 0.1, 1, None) == 3        # g > 128
    # B * Hq past 2^31 - 1 (one combine CTA per row), refused before the workspace is sized
    assert lib.attn_decode_fp8(*dargs, wdec, 65535, 32769, 32769, 128, 128, 0.1, 1, None) == 3
    assert lib.attn_decode_fp8(*dargs, wdec, 65535, 32768, 256, 128, 64, 0.1, 1, None) == 7   # fits: workspace next
    # fused RoPE producer: the tables are required and aligned
    assert lib.attn_quantize_fp8_rope(P(16), 0, P(16), P(16), 1, 1, 8, 64, None, P(16), None, None) == 1
    assert lib.attn_quantize_fp8_rope(P(16), 0, P(16), P(16), 1, 1, 8, 64, P(16), P(20), None, None) == 2
    assert lib.attn_quantize_fp8_rope(P(16), 0, P(16), P(16), 1, 1, 8, 96, P(16), P(16), None, None) == 4
    # quantiser: head dim and dtype
    assert lib.attn_quantize_fp8(P(16), 0, P(16), P(16), 1, 1, 8, 32, None, None) == 4
    assert lib.attn_quantize_fp8(P(16), 2, P(16), P(16), 1, 1, 8, 64, None, None) == 6
    # FP8 forward: scales are required and aligned; head dim and GQA as attn_fwd
    f8 = [P(16)] * 3
    assert lib.attn_fwd_fp8(*f8, None, P(16), P(16), P(16), P(16), 1, 2, 1, 8, 128, 0.1, 0, None) == 1
    assert lib.attn_fwd_fp8(*f8, P(16), P(20), P(16), P(16), P(16), 1, 2, 1, 8, 128, 0.1, 0, None) == 2
    assert lib.attn_fwd_fp8(*f8, P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 0, 128, 0.1, 0, None) == 3
    assert lib.attn_fwd_fp8(*f8, P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 8, 96, 0.1, 0, None) == 4
    assert lib.attn_fwd_fp8(*f8, P(16), P(16), P(16), P(16), P(16), 1, 3, 2, 8, 128, 0.1, 0, None) == 5
    # FP8 with a key window: bounds below -1 refused, the rest as attn_fwd_fp8
    assert lib.attn_fwd_fp8_window(*f8, P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 8, 128, 0.1, -2, 0, None) == 3
    assert lib.attn_fwd_fp8_window(*f8, P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 8, 128, 0.1, 4, -3, None) == 3
    assert lib.attn_fwd_fp8_window(*f8, None, P(16), P(16), P(16), P(16), 1, 2, 1, 8, 128, 0.1, 4, 4, None) == 1
    assert lib.attn_fwd_fp8_window(*f8, P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 8, 96, 0.1, 4, 4, None) == 4
    assert lib.attn_fwd_fp8_window(*f8, P(16), P(16), P(16), P(16), P(16), 1, 3, 2, 8, 128, 0.1, 4, 4, None) == 5
    # packed FP8: cu_seqlens required and aligned, nseq / T / max_seqlen, head dim, dtype, GQA
    assert lib.attn_quantize_fp8_varlen(P(16), 0, P(16), P(16), None, 2, 10, 5, 1, 64, None, None) == 1
    assert lib.attn_quantize_fp8_varlen(P(16), 0, P(16), P(16), P(24), 2, 10, 5, 1, 64, None, None) == 2
    assert lib.attn_quantize_fp8_varlen(P(16), 0, P(16), P(16), P(16), 2, 10, 11, 1, 64, None, None) == 3
    assert lib.attn_quantize_fp8_varlen(P(16), 0, P(16), P(16), P(16), 0, 10, 5, 1, 64, None, None) == 3
    assert lib.attn_quantize_fp8_varlen(P(16), 0, P(16), P(16), P(16), 2, 10, 5, 1, 32, None, None) == 4
    assert lib.attn_quantize_fp8_varlen(P(16), 2, P(16), P(16), P(16), 2, 10, 5, 1, 64, None, None) == 6
    v8 = [P(16)] * 8
    assert lib.attn_fwd_fp8_varlen(*v8, None, 2, 10, 5, 2, 1, 128, 0.1, 0, None) == 1
    assert lib.attn_fwd_fp8_varlen(*v8, P(16), 2, 10, 11, 2, 1, 128, 0.1, 0, None) == 3
    assert lib.attn_fwd_fp8_varlen(*v8, P(16), 2, 10, 5, 2, 1, 96, 0.1, 0, None) == 4
    assert lib.attn_fwd_fp8_varlen(*v8, P(16), 2, 10, 5, 3, 2, 128, 0.1, 0, None) == 5
    # varlen backward: cu_seqlens, sequence counts and the workspace are checked
    wv = binding.attn_bwd_varlen_workspace_size(10, 2, 1, 128)
    vargs = [P(16)] * 9
    assert lib.attn_bwd_varlen(*vargs, P(16), wv, None, 2, 10, 5, 2, 1, 128, 0.1, 0, 0, None) == 1
    assert lib.attn_bwd_varlen(*vargs, P(16), wv, P(16), 0, 10, 5, 2, 1, 128, 0.1, 0, 0, None) == 3
    assert lib.attn_bwd_varlen(*vargs, P(16), wv, P(16), 2, 10, 11, 2, 1, 128, 0.1, 0, 0, None) == 3
    assert lib.attn_bwd_varlen(*vargs, P(16), wv - 1, P(16), 2, 10, 5, 2, 1, 128, 0.1, 0, 0, None) == 7
    # backward: workspace must be present and large enough
    ws = binding.attn_bwd_workspace_size(1, 2, 1, 8, 128)
    args = [P(16)] * 9
    assert lib.attn_bwd(*args, None, ws, 1, 2, 1, 8, 128, 0.1, 0, 0, None) == 1
    assert lib.attn_bwd(*args, P(16), ws - 1, 1, 2, 1, 8, 128, 0.1, 0, 0, None) == 7
    assert lib.attn_bwd(*args, P(16), ws, 1, 2, 1, 8, 96, 0.1, 0, 0, None) == 4   # backward: d = 64, 128, 256
    assert lib.attn_bwd(*args, P(16), ws, 1, 2, 1, 8, 64, 0.1, 0, 0, None) == 11  # d = 64 valid: no device here
    # sliding window: bounds are -1 (unbounded) or >= 0
    assert lib.attn_fwd_window(P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 8, 64, 0.1, -2, 0, 0, None) == 3
    assert lib.attn_fwd_window(P(16), P(16), P(16), P(16), P(16), 1, 2, 1, 8, 64, 0.1, 4, -3, 0, None) == 3
    assert lib.attn_fwd_window(None, P(16), P(16), P(16), P(16), 1, 2, 1, 8, 64, 0.1, 4, 0, 0, None) == 1
    assert lib.attn_bwd_window(*args, P(16), ws, 1, 2, 1, 8, 128, 0.1, -5, 0, 0, None) == 3
    assert lib.attn_bwd_window(*args, P(16), ws - 1, 1, 2, 1, 8, 128, 0.1, 3, 0, 0, None) == 7
    # deterministic backward: its own (D-only) workspace, d = 64 or 128, window bounds
    wd = binding.attn_bwd_deterministic_workspace_size(1, 2, 1, 8, 128)
    assert wd == 256
    assert lib.attn_bwd_deterministic(*args, P(16), wd - 1, 1, 2, 1, 8, 128, 0.1, -1, -1, 0, None) == 7
    assert lib.attn_bwd_deterministic(*args, P(16), wd, 1, 2, 1, 8, 256, 0.1, -1, -1, 0, None) == 4
    assert lib.attn_bwd_deterministic(*args, P(16), wd, 1, 2, 1, 8, 96, 0.1, -1, -1, 0, None) == 4
    assert lib.attn_bwd_deterministic(*args, P(16), wd, 1, 2, 1, 8, 128, 0.1, -3, 0, 0, None) == 3


def test_workspace_size_arithmetic():
    up = lambda x: (x + 255) // 256 * 256
    B, Hq, N, d = 2, 32, 8192, 128
    assert binding.attn_bwd_workspace_size(B, Hq, 8, N, d) == up(B * Hq * N * d * 4) + up(B * Hq * N * 4)
    assert binding.attn_bwd_varlen_workspace_size(1000, 4, 2, 64) == up(1000 * 4 * 64 * 4) + up(1000 * 4 * 4)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_fails_loudly(lib):
    assert _fwd(lib) == 11                          # ATTN_ERR_NODEVICE, nothing launched


C_CLIENT = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include "libattn.h"

int main(void) {
  int bad = 0;
  for (int s = ATTN_OK; s <= ATTN_ERR_NODEVICE; ++s) {
    const char* n = attn_status_string((attn_status)s);
    printf("%d %s\n", s, n ? n : "(null)");
    if (!n || strncmp(n, "ATTN_", 5) != 0) bad = 1;
  }
  printf("version %s\n", attn_version());
  /* argument checks return before any device work; host memory stands in for device pointers */
  static char buf[64];
  void* p = (void*)(((uintptr_t)buf + 15) & ~(uintptr_t)15);
  if (attn_fwd(NULL, p, p, p, (float*)p, 1, 2, 1, 8, 64, 0.125f, 0, ATTN_BF16, NULL) != ATTN_ERR_NULL) bad = 2;
  if (attn_fwd(p, p, p, p, (float*)p, 1, 2, 1, 8, 96, 0.125f, 0, ATTN_BF16, NULL) != ATTN_ERR_HEADDIM) bad = 3;
  if (attn_fwd(p, p, p, p, (float*)p, 1, 3, 2, 8, 64, 0.125f, 0, ATTN_BF16, NULL) != ATTN_ERR_GQA) bad = 4;
  if (attn_fwd_fp8_kv_tile(128) != 128) bad = 5;
  if (attn_bwd_workspace_size(2, 32, 8, 8192, 128) != (size_t)2 * 32 * 8192 * 128 * 4 + (size_t)2 * 32 * 8192 * 4)
    bad = 6;
  if (ATTN_BWD_NOALLOC_MAX_BYTES != 32u * 1024u * 1024u) bad = 7;
  printf("%s %d\n", bad ? "FAIL" : "OK", bad);
  return bad;
}
"""


def test_plain_c_client_compiles_links_and_runs(lib, tmp_path):
    """The header is plain C (gcc -std=c11 -Wall -Werror) and a C program
    links against libattn.so and gets the documented answers without a GPU."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    from exact_attention_73_gb300 import build
    src, exe = tmp_path / "client.c", tmp_path / "client"
    src.write_text(C_CLIENT)
    libdir = os.path.dirname(build.LIB)
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                        "-o", str(exe), f"-L{libdir}", f"-l:{os.path.basename(build.LIB)}", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.splitlines()
    for code, name in binding.STATUS.items():
        assert lines[code].split()[1].rstrip(":") == name, lines[code]
    assert lines[-1] == "OK 0"
