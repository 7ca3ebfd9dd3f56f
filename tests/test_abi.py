"""The C-ABI library builds, loads and exports what include/pagedkv.h declares.

No kernel is launched here (these run without a GPU): only host-side sizes,
strings and argument checks that return before any CUDA call.
"""

import ctypes
import os
import re

import pytest

import oracle
from paged_kv_cache_45_gb300 import build as pk_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    path = pk_build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for fn in ("pa_kv_append", "pa_decode", "pa_decode_splitk_reduce"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from paged_kv_cache_45_gb300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


def test_status_strings_and_version():
    from paged_kv_cache_45_gb300 import binding as b
    assert b.pa_status_str(0) == "PA_OK"
    assert b.pa_status_str(-1) == "PA_ERR_INVALID_ARG"
    assert b.pa_status_str(-5) == "PA_ERR_DEVICE"
    assert b.pa_status_str(99) == "PA_ERR_UNKNOWN"
    assert "sm_103a" in b.pa_version()


def test_sizes_match_the_oracle_formula():
    from paged_kv_cache_45_gb300 import binding as b
    for args in [(32, 8, 128, 2), (80, 8, 128, 2), (80, 8, 128, 1), (1, 8, 128, 2)]:
        assert b.pa_kv_bytes_per_token(*args) == oracle.kv_bytes_per_token(*args)
    assert b.pa_decode_num_splits(131072, 4096) == 32
    assert b.pa_decode_num_splits(131073, 4096) == 33
    assert b.pa_decode_num_splits(0, 4096) == 0
    assert b.pa_decode_num_splits(100, 0) == 0
    rows = 4 * 32 * 32
    assert b.pa_decode_workspace_bytes(4, 32, 128, 32) == rows * 128 * 4 + rows * 4


def test_bad_arguments_are_rejected_before_any_launch(lib):
    lib.pa_decode.restype = ctypes.c_int32
    lib.pa_kv_append.restype = ctypes.c_int32
    lib.pa_decode_splitk_reduce.restype = ctypes.c_int32
    P = ctypes.c_void_p
    fake = P(4096)           # never dereferenced: checks fail first
    odd = P(4098)            # not 16-byte aligned

    def decode(q=fake, k=fake, v=fake, bt=fake, mb=4, cl=fake, B=2, hq=8, hkv=2, d=128, bs=16,
               nb=16, scale=0.1, split=0, ms=0, po=None, pl=None, out=fake):
        return lib.pa_decode(q, k, v, bt, ctypes.c_int32(mb), cl, ctypes.c_int32(B),
                             ctypes.c_int32(hq), ctypes.c_int32(hkv), ctypes.c_int32(d),
                             ctypes.c_int32(bs), ctypes.c_int32(nb), ctypes.c_float(scale),
                             ctypes.c_int32(split), ctypes.c_int32(ms), po, pl, out, None)

    assert decode(q=None) == -1
    assert decode(hq=7, hkv=2) == -1           # heads do not group
    assert decode(hq=32, hkv=2) == -2          # group of 16: not built
    assert decode(d=96) == -2                  # head_dim
    assert decode(bs=12) == -2                 # block size not a power of two
    assert decode(q=odd) == -1                 # alignment
    assert decode(split=24, ms=4, po=fake, pl=fake) == -1   # split not a multiple of 16
    assert decode(split=32, ms=4) == -4        # split without partial buffers
    assert decode(split=32, ms=0, po=fake, pl=fake) == -1
    assert decode(nb=1 << 27, bs=32) == -1     # pool rows overflow int32
    assert decode(scale=float("nan")) == -1
    assert decode(B=0) == 0                    # nothing to do

    lib.pa_decode_balanced.restype = ctypes.c_int32

    def balanced(q=fake, B=2, hq=8, hkv=2, d=128, bs=16, ws=fake, ws_bytes=1 << 20):
        return lib.pa_decode_balanced(q, fake, fake, fake, ctypes.c_int32(4), fake,
                                      ctypes.c_int32(B), ctypes.c_int32(hq), ctypes.c_int32(hkv),
                                      ctypes.c_int32(d), ctypes.c_int32(bs), ctypes.c_int32(16),
                                      ctypes.c_float(0.1), ws, ctypes.c_size_t(ws_bytes), fake,
                                      None)

    assert balanced(q=None) == -1
    assert balanced(hq=7) == -1
    assert balanced(d=80) == -2
    assert balanced(bs=3) == -2
    assert balanced(B=0) == 0

    T = ctypes.c_int32
    assert lib.pa_kv_append(fake, fake, fake, T(4), None, fake, T(8), T(16), T(2), T(64), None) == -1
    assert lib.pa_kv_append(fake, fake, fake, T(4), fake, fake, T(8), T(16), T(2), T(60), None) == -2
    assert lib.pa_kv_append(odd, fake, fake, T(4), fake, fake, T(8), T(16), T(2), T(64), None) == -1
    assert lib.pa_kv_append(fake, fake, fake, T(0), fake, fake, T(8), T(16), T(2), T(64), None) == 0

    assert lib.pa_decode_splitk_reduce(fake, fake, fake, T(2), T(8), T(128), T(0), T(4), fake,
                                       None) == -1
    assert lib.pa_decode_splitk_reduce(fake, fake, fake, T(2), T(8), T(80), T(16), T(4), fake,
                                       None) == -2


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "pagedkv.h"

int main(void) {
  if (strcmp(pa_status_str(PA_OK), "PA_OK") != 0) return 1;
  if (pa_kv_bytes_per_token(80, 8, 128, 2) != 327680) return 2;
  if (pa_decode_num_splits(131073, 4096) != 33) return 3;
  pa_prefix_cache* pc = NULL;
  if (pa_prefix_cache_create(64, 4, &pc) != PA_OK || !pc) return 4;
  int32_t toks[10];
  for (int i = 0; i < 10; ++i) toks[i] = 100 + i;
  int64_t sid = 0;
  int32_t cached = -1;
  if (pa_prefix_admit(pc, toks, 10, &sid, &cached) != PA_OK || sid <= 0 || cached != 0) return 5;
  int64_t slots[10];
  int32_t src[4], dst[4], nc = -1;
  if (pa_prefix_write_slots(pc, sid, 0, 10, slots, src, dst, 4, &nc) != PA_OK || nc != 0)
    return 6;
  for (int p = 0; p < 10; ++p)  /* fresh blocks lowest id first: 1, 2, 3 */
    if (slots[p] != (int64_t)(1 + p / 4) * 4 + p % 4) return 7;
  int32_t table[8], lens[1];
  if (pa_prefix_tables(pc, &sid, 1, table, 8, lens) != PA_OK || lens[0] != 10 ||
      table[0] != 1 || table[2] != 3 || table[3] != 0)
    return 8;
  int32_t free_blocks = -1, cached_blocks = -1, used = -1;
  if (pa_prefix_stats(pc, &free_blocks, &cached_blocks, &used) != PA_OK || free_blocks != 60 ||
      used != 3)
    return 9;
  if (pa_prefix_discard(pc, &sid, 1) != PA_OK) return 10;
  if (pa_prefix_stats(pc, &free_blocks, &cached_blocks, &used) != PA_OK || free_blocks != 63 ||
      used != 0)
    return 11;
  pa_prefix_cache_destroy(pc);
  if (pa_kv_append(NULL, NULL, NULL, 1, NULL, NULL, 16, 16, 8, 128, NULL) != PA_ERR_INVALID_ARG)
    return 12;
  printf("ok %s\n", pa_version());
  return 0;
}
"""


def test_header_compiles_as_c_and_the_library_links(tmp_path):
    # the boundary is a plain C ABI: a C11 program includes the header, links
    # the library and makes host-only calls (no GPU needed)
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib_path = pk_build.build()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    lib_dir = os.path.dirname(lib_path)
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", lib_dir,
                        "-l:" + os.path.basename(lib_path), "-Wl,-rpath," + lib_dir],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.startswith("ok ") and "sm_103a" in r.stdout
