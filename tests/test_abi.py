"""The C-ABI library loads without a GPU, exports every entry point that
include/dsa.h declares, and rejects bad host-side arguments before touching
the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DSA_API\s+[\w\s\*]+?\b((?:dsa|indexshare)_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def dsa():
    import dsa_indexer_indexshare_gb300 as m
    return m


def test_header_declares_the_hot_path_calls():
    fns = declared_functions()
    for name in ("dsa_indexer_scores", "dsa_topk", "dsa_sparse_mla_attn",
                 "indexshare_group_forward", "dsa_fp8_quantize"):
        assert name in fns


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++11")])
def test_header_is_plain_c(lang, std, tmp_path):
    """The boundary header compiles on its own, as C99 and as C++, with no
    CUDA or torch headers (a C caller needs nothing else), and a C program
    can take the address of every declared entry point."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-x", lang, HEADER], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    src = tmp_path / ("use.c" if lang == "c" else "use.cc")
    body = "\n".join(f"  (void)&{f};" for f in declared_functions())
    src.write_text(f'#include "{HEADER}"\nint main(void) {{\n{body}\n  return 0;\n}}\n')
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Werror", "-fsyntax-only", str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(dsa):
    lib = ctypes.CDLL(dsa.LIB_PATH)
    missing = [f for f in declared_functions() if not hasattr(lib, f)]
    assert not missing, missing


def _batch(dsa, num_q=4, max_q=4, max_len=256, ptr=256):
    return dsa._Batch(1, num_q, max_q, max_len, ctypes.c_void_p(ptr), ctypes.c_void_p(ptr),
                      ctypes.c_void_p(ptr))


def test_argument_errors_without_a_device(dsa):
    L = dsa.lib
    fake = ctypes.c_void_p(4096)
    b = _batch(dsa)
    # max_len not a multiple of 128
    bad = _batch(dsa, max_len=200)
    assert L.dsa_topk(fake, ctypes.byref(bad), 16, fake, fake, 256, None) == dsa.DSA_ERR_INVALID_ARG
    assert b"multiple of 128" in L.dsa_last_error_string()
    # k out of range
    assert L.dsa_topk(fake, ctypes.byref(b), 0, fake, fake, 256, None) == dsa.DSA_ERR_UNSUPPORTED
    # workspace too small / misaligned
    assert L.dsa_topk(fake, ctypes.byref(b), 16, fake, fake, 8, None) == dsa.DSA_ERR_WORKSPACE
    assert L.dsa_topk(fake, ctypes.byref(b), 16, fake, ctypes.c_void_p(4097), 256,
                      None) == dsa.DSA_ERR_WORKSPACE
    # unsupported head count
    assert L.dsa_sparse_mla_attn(fake, fake, fake, 100, fake, 64, 32, 0.0625, ctypes.byref(b), fake,
                                 None, fake, 256, None) == dsa.DSA_ERR_UNSUPPORTED
    # misaligned operand
    assert L.dsa_sparse_mla_attn(ctypes.c_void_p(4098), fake, fake, 100, fake, 64, 64, 0.0625,
                                 ctypes.byref(b), fake, None, fake, 256,
                                 None) == dsa.DSA_ERR_INVALID_ARG
    # FP8 indexer without scales
    assert L.dsa_indexer_scores(fake, None, fake, fake, None, 100, dsa.DSA_FP8_E4M3, ctypes.byref(b),
                                fake, fake, 256, None) == dsa.DSA_ERR_INVALID_ARG
    # NULL batch
    assert L.dsa_indexer_scores(fake, None, fake, fake, None, 100, 0, None, fake, fake, 256,
                                None) == dsa.DSA_ERR_INVALID_ARG


def test_group_layer_string_is_validated(dsa):
    L = dsa.lib
    b = _batch(dsa)
    arr = (ctypes.c_void_p * 4)(*[4096] * 4)
    pp = ctypes.cast(arr, dsa._PP)
    for types, ok in ((b"SFSS", False), (b"FXSS", False), (b"", False)):
        g = dsa._Group(types, 64, 2048, 0.0625, 0, 100, 100, pp, pp, pp, pp, None, pp, None, pp, pp,
                       None)
        st = L.indexshare_group_forward(ctypes.byref(g), ctypes.byref(b), ctypes.c_void_p(4096),
                                        ctypes.c_void_p(4096), 1 << 30, None)
        assert st == dsa.DSA_ERR_INVALID_ARG
    # a valid string with a workspace below the required size
    g = dsa._Group(b"FSSS", 64, 2048, 0.0625, 0, 100, 100, pp, pp, pp, pp, None, pp, None, pp, pp,
                   None)
    need = L.dsa_group_workspace_size(ctypes.byref(g), ctypes.byref(b))
    assert need >= 256 + 4 * 256 * 4
    st = L.indexshare_group_forward(ctypes.byref(g), ctypes.byref(b), ctypes.c_void_p(4096),
                                    ctypes.c_void_p(4096), need - 256, None)
    assert st == dsa.DSA_ERR_WORKSPACE


def test_launch_counters_and_timeout_setter(dsa):
    dsa.launch_counts_reset()
    assert set(dsa.launch_counts().values()) == {0}
    dsa.set_wait_timeout_ns(2_000_000_000)


def test_append_and_paged_argument_errors_without_a_device(dsa):
    L = dsa.lib
    fake = ctypes.c_void_p(4096)
    b = _batch(dsa)
    freq = (ctypes.c_double * 32)(*([1.0] * 32))
    # no rotary frequencies
    assert L.dsa_indexer_append_keys(fake, fake, fake, 4, ctypes.byref(b), dsa.DSA_BF16, None, fake,
                                     None, 100, fake, 256, None) == dsa.DSA_ERR_INVALID_ARG
    assert b"inv_freq" in L.dsa_last_error_string()
    # negative count, unknown dtype, FP8 without scales, misaligned keys
    assert L.dsa_indexer_append_keys(fake, fake, fake, -1, ctypes.byref(b), dsa.DSA_BF16, freq,
                                     fake, None, 100, fake, 256, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_indexer_append_keys(fake, fake, fake, 4, ctypes.byref(b), 7, freq, fake, None, 100,
                                     fake, 256, None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_indexer_append_keys(fake, fake, fake, 4, ctypes.byref(b), dsa.DSA_FP8_E4M3, freq,
                                     fake, None, 100, fake, 256, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_indexer_append_keys(ctypes.c_void_p(4100), fake, fake, 4, ctypes.byref(b),
                                     dsa.DSA_BF16, freq, fake, None, 100, fake, 256,
                                     None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_indexer_prepare_queries(fake, ctypes.byref(b), dsa.DSA_FP8_E4M3, freq, fake, None,
                                         fake, 256, None) == dsa.DSA_ERR_INVALID_ARG
    # paged layout: block size not a power of two >= 128, table too short for max_len
    for rows, per_seq in ((384, 4), (64, 4), (128, 1)):
        pb = dsa._Batch(1, 4, 4, 256, fake, fake, None, fake, rows, per_seq)
        assert L.dsa_topk(fake, ctypes.byref(pb), 16, fake, fake, 256,
                          None) == dsa.DSA_ERR_INVALID_ARG
    # a paged batch needs no seq_row0; a contiguous one does
    ok = dsa._Batch(1, 0, 0, 256, fake, fake, None, fake, 128, 2)
    assert L.dsa_topk(fake, ctypes.byref(ok), 16, fake, fake, 256, None) == dsa.DSA_OK
    nob = dsa._Batch(1, 0, 0, 256, fake, fake, None)
    assert L.dsa_topk(fake, ctypes.byref(nob), 16, fake, fake, 256, None) == dsa.DSA_ERR_INVALID_ARG


def test_hot_argument_errors_without_a_device(dsa):
    L = dsa.lib
    fake = ctypes.c_void_p(4096)
    b = _batch(dsa, max_len=256)
    ws = ctypes.c_void_p(1 << 20)

    def hot(slots=64, max_pos=256, arrays=True):
        p = fake if arrays else None
        return dsa._Hot(slots, max_pos, p, p, p, p, p, p)

    ok = hot()
    assert L.dsa_hot_plan(fake, 16, ctypes.byref(b), ctypes.byref(hot(slots=0)), 0, fake, ws, 256,
                          None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_hot_plan(fake, 16, ctypes.byref(b), ctypes.byref(hot(slots=dsa.HOT_MAX_SLOTS + 1)),
                          0, fake, ws, 256, None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_hot_plan(fake, 16, ctypes.byref(b), ctypes.byref(hot(max_pos=128)), 0, fake, ws,
                          256, None) == dsa.DSA_ERR_INVALID_ARG
    assert b"max_pos" in L.dsa_last_error_string()
    assert L.dsa_hot_plan(fake, 16, ctypes.byref(b), ctypes.byref(hot(arrays=False)), 0, fake, ws,
                          256, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_hot_plan(fake, 16, ctypes.byref(b), ctypes.byref(ok), -1, fake, ws, 256,
                          None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_hot_plan(fake, 16, ctypes.byref(b), None, 0, fake, ws, 256,
                          None) == dsa.DSA_ERR_INVALID_ARG
    # cold caches: host memory CUDA does not know (pageable) is refused
    host = (ctypes.c_uint8 * 4096)()
    addr = (ctypes.addressof(host) + 15) & ~15
    cold = (ctypes.c_void_p * 1)(addr)
    hotp = (ctypes.c_void_p * 1)(4096)
    assert L.dsa_hot_fetch(ctypes.byref(ok), ctypes.byref(b), 1, ctypes.cast(cold, dsa._PP), 2,
                           ctypes.cast(hotp, dsa._PP), 64, dsa.DSA_BF16, ws, 256,
                           None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_hot_fetch(ctypes.byref(ok), ctypes.byref(b), 1, ctypes.cast(cold, dsa._PP), 2,
                           ctypes.cast(hotp, dsa._PP), 64, 7, ws, 256, None) == dsa.DSA_ERR_UNSUPPORTED
    # hot arrays smaller than num_seqs * hot_slots rows
    assert L.dsa_hot_fetch(ctypes.byref(ok), ctypes.byref(b), 1, ctypes.cast(cold, dsa._PP), 2,
                           ctypes.cast(hotp, dsa._PP), 63, dsa.DSA_BF16, ws, 256,
                           None) == dsa.DSA_ERR_INVALID_ARG
    assert b"hot_rows" in L.dsa_last_error_string()
    # rows-mode attention: FP8 rows need 64 heads
    assert L.dsa_sparse_mla_attn_rows(fake, fake, fake, 100, dsa.DSA_FP8_E4M3, fake, 64, 16, 0.0625,
                                      ctypes.byref(b), fake, None, ws, 256,
                                      None) == dsa.DSA_ERR_UNSUPPORTED


def test_hot_touch_argument_errors_without_a_device(dsa):
    L = dsa.lib
    host = (ctypes.c_uint8 * 4096)()
    cold = (ctypes.c_void_p * 1)((ctypes.addressof(host) + 15) & ~15)
    pp = ctypes.cast(cold, dsa._PP)
    assert L.dsa_hot_touch(1, pp, 1024, 24, None) == dsa.DSA_ERR_INVALID_ARG  # stride % 16
    assert L.dsa_hot_touch(1, pp, 0, 4096, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_hot_touch(1, None, 1024, 4096, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_hot_touch(0, None, 1024, 4096, None) == dsa.DSA_OK
    # pageable host memory is refused
    assert L.dsa_hot_touch(1, pp, 1024, 4096, None) == dsa.DSA_ERR_INVALID_ARG


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "dsa.h"

int main(void) {
  dsa_batch_t b;
  memset(&b, 0, sizeof b);
  b.num_seqs = 1; b.num_q = 4; b.max_q = 4; b.max_len = 200;  /* not a multiple of 128 */
  b.q_start = (const int32_t*)256; b.q_pos = (const int32_t*)256; b.seq_row0 = (const int64_t*)256;
  void* p = (void*)4096;
  if (dsa_topk((const float*)p, &b, 16, (int32_t*)p, p, 256, NULL) != DSA_ERR_INVALID_ARG) return 1;
  if (strstr(dsa_last_error_string(), "multiple of 128") == NULL) return 2;
  b.max_len = 256;
  if (dsa_topk((const float*)p, &b, 0, (int32_t*)p, p, 256, NULL) != DSA_ERR_UNSUPPORTED) return 3;
  if (dsa_sparse_mla_attn(p, p, p, 100, (const int32_t*)p, 64, 32, 0.0625f, &b, p, NULL, p, 256,
                          NULL) != DSA_ERR_UNSUPPORTED) return 4;
  if (dsa_status_bytes() != 256) return 5;
  dsa_hot_t h;
  memset(&h, 0, sizeof h);
  if (dsa_hot_plan((const int32_t*)p, 16, &b, &h, 0, (int32_t*)p, p, 256, NULL) != DSA_ERR_UNSUPPORTED)
    return 6;
  printf("ok\n");
  return 0;
}
"""


def test_a_c_program_links_and_gets_argument_errors(dsa, tmp_path):
    """A C caller compiled against include/dsa.h and linked to libdsa.so
    gets the documented status codes from host-side argument checks (no
    kernel is launched)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(dsa.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                        "-o", str(exe), "-L", libdir, "-ldsa", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
