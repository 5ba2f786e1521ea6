"""The C-ABI library loads and exports every function include/pkv.h declares,
and rejects bad host-side arguments without launching anything.  CPU only:
no call here reaches a kernel (each returns before any launch)."""

import ctypes
import os
import subprocess

import pytest

import paged_kv_cache_304_gb300 as pkv

LIB = pkv.LIB_PATH


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from paged_kv_cache_304_gb300 import build
        build.build()
    return pkv.load()


def test_header_declares_the_three_calls():
    names = pkv.exported_functions()
    for n in ("pkv_kv_cache_write", "pkv_paged_attn_decode", "pkv_paged_attn_prefill",
              "pkv_paged_attn_decode_fused_write"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    declared = set(pkv.exported_functions())
    assert declared <= exported, declared - exported
    for name in declared:
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.pkv_status_string(code)
    assert lib.pkv_version() >= 100


def test_kv_write_argument_errors(lib):
    vp = ctypes.c_void_p
    fake = vp(0x1000)  # never dereferenced: every call below fails validation first
    # negative token count
    assert lib.pkv_kv_cache_write(fake, 1024, fake, 1024, fake, -1, fake, fake, 4, 256, 8, 128, None) == -2
    # stride smaller than a row
    assert lib.pkv_kv_cache_write(fake, 512, fake, 1024, fake, 4, fake, fake, 4, 256, 8, 128, None) == -2
    # null pointer
    assert lib.pkv_kv_cache_write(None, 1024, fake, 1024, fake, 4, fake, fake, 4, 256, 8, 128, None) == -1
    # misaligned pointer
    assert lib.pkv_kv_cache_write(vp(0x1002), 1024, fake, 1024, fake, 4, fake, fake, 4, 256, 8, 128, None) == -6
    # zero tokens is a no-op
    assert lib.pkv_kv_cache_write(None, 1024, None, 1024, None, 0, None, None, 4, 256, 8, 128, None) == 0


def test_decode_argument_errors(lib):
    vp = ctypes.c_void_p
    f = vp(0x1000)
    args = dict(maxb=4, B=2, hq=16, hkv=8, d=128, bs=256, nb=8, maxctx=1024, scale=0.088)

    def call(**kw):
        a = {**args, **kw}
        return lib.pkv_paged_attn_decode(f, f, f, f, f, a["maxb"], a["B"], a["hq"], a["hkv"], a["d"], a["bs"],
                                         a["nb"], a["maxctx"], a["scale"], f, kw.get("ws", f), kw.get("wsb", 0),
                                         None)

    assert call(d=64) == -3          # head_dim 64 unsupported
    assert call(bs=16) == -3         # block_size 16 unsupported
    assert call(hq=12) == -2         # not a multiple of the kv heads
    assert call(hkv=16, hq=32) == -3  # more than 8 kv heads
    assert call(scale=0.0) == -2
    assert call(B=-1) == -2
    assert call(B=0) == 0            # empty batch is a no-op


def test_prefill_argument_errors(lib):
    vp = ctypes.c_void_p
    f = vp(0x1000)
    r = lib.pkv_paged_attn_prefill(f, f, f, f, f, f, 4, 2, 100, 64, 300, 16, 8, 64, 256, 8, 0.1, f, None)
    assert r == -3  # head_dim 64


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(pkv.PkvLibraryError):
        pkv.load(str(tmp_path / "missing.so"))


C_CALLER = r"""
#include <stdio.h>
#include "pkv.h"

/* A plain C caller of the library: the header is C, and the calls below
   fail host-side validation (no device is touched). */
int main(void) {
  const void* fake = (const void*)0x1000;
  int rc;
  if (pkv_version() < 100) return 1;
  if (!pkv_status_string(PKV_ERR_NULL)) return 2;
  rc = pkv_kv_cache_write(NULL, 1024, fake, 1024, (const int32_t*)fake, 4, (pkv_bf16*)fake, (pkv_bf16*)fake, 4,
                          256, 8, 128, NULL);
  if (rc != PKV_ERR_NULL) return 3;
  rc = pkv_paged_attn_prefill(fake, fake, fake, (const int32_t*)fake, (const int32_t*)fake, (const int32_t*)fake,
                              8, 1, 16, 16, 16, 16, 8, 96, 256, 4, 0.088f, (pkv_bf16*)fake, NULL);
  if (rc != PKV_ERR_UNSUPPORTED) return 4;
  printf("ok %d\n", pkv_version());
  return 0;
}
"""


def test_plain_c_caller_links_and_runs(lib, tmp_path):
    """The boundary works from C: compile a C99 program against include/pkv.h,
    link it to libpkv.so and run it (argument-validation paths only)."""
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    libdir = os.path.dirname(LIB)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", inc, str(src), "-o", str(exe),
                    "-L", libdir, "-lpkv", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert out.stdout.startswith("ok ")
