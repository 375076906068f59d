"""Host-side checks of the C interface that need no GPU.

The library is loaded with ctypes, every function declared in include/gqa.h
must be exported, and argument validation must reject bad calls with the
documented status before any CUDA call is made (so these run on a machine
without a device or driver).
"""

import ctypes
import os
import re

import pytest

from grouped_query_attention_10_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa.h")

FAKE = 1 << 20        # a 16-byte-aligned non-null address; never dereferenced
MISALIGNED = FAKE + 8


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


@pytest.fixture(scope="module")
def lib():
    return binding.load_library()


def test_header_declares_the_three_entry_points():
    names = _declared_functions()
    for n in ("gqa_prefill_fwd", "gqa_decode_fwd", "kv_cache_append",
              "gqa_decode_workspace_bytes", "gqa_status_string", "gqa_version"):
        assert n in names, names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"{n} declared in gqa.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.gqa_version() == 100
    for code in range(0, 11):
        s = binding.status_string(code)
        assert s.startswith("GQA_")
    assert binding.status_string(99) == "GQA_ERR_UNKNOWN"


def _prefill(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, o_dtype=0, lse=None, B=1, L=128, h_q=8,
             g=2, d=64, scale=0.125, causal=1, status=None):
    return lib.gqa_prefill_fwd(q, k, v, o, o_dtype, lse, B, L, h_q, g, d, scale, causal,
                               status, None)


def test_prefill_validation(lib):
    assert _prefill(lib, q=None) == binding.GQA_ERR_NULL
    assert _prefill(lib, o=None) == binding.GQA_ERR_NULL
    assert _prefill(lib, B=0) == binding.GQA_ERR_SHAPE
    assert _prefill(lib, L=0) == binding.GQA_ERR_SHAPE
    assert _prefill(lib, h_q=8, g=3) == binding.GQA_ERR_SHAPE    # g does not divide h_q
    assert _prefill(lib, h_q=12, g=2) == binding.GQA_ERR_SHAPE   # group size 6 not a power of 2
    assert _prefill(lib, h_q=256, g=1) == binding.GQA_ERR_SHAPE  # group size > 128
    assert _prefill(lib, d=96) == binding.GQA_ERR_SHAPE
    assert _prefill(lib, o_dtype=7) == binding.GQA_ERR_SHAPE
    assert _prefill(lib, scale=0.0) == binding.GQA_ERR_SHAPE
    assert _prefill(lib, scale=float("nan")) == binding.GQA_ERR_SHAPE
    assert _prefill(lib, q=MISALIGNED) == binding.GQA_ERR_ALIGN
    assert _prefill(lib, o=MISALIGNED) == binding.GQA_ERR_ALIGN
    assert _prefill(lib, lse=FAKE + 2) == binding.GQA_ERR_ALIGN


def _decode(lib, q=FAKE, kc=FAKE, vc=FAKE, lens=FAKE, o=FAKE, o_dtype=0, lse=None, B=4,
            h_q=32, g=8, d=128, S_max=1024, scale=0.088, ws=FAKE, ws_bytes=None, status=None):
    if ws_bytes is None:
        ws_bytes = lib.gqa_decode_workspace_bytes(B, h_q, g, d, S_max)
    return lib.gqa_decode_fwd(q, kc, vc, lens, o, o_dtype, lse, B, h_q, g, d, S_max, scale,
                              ws, ws_bytes, status, None)


def test_decode_workspace_bytes(lib):
    n = lib.gqa_decode_workspace_bytes(64, 32, 8, 128, 8192)
    assert n > 0 and n % 4 == 0
    assert lib.gqa_decode_workspace_bytes(64, 32, 8, 96, 8192) == 0
    assert lib.gqa_decode_workspace_bytes(0, 32, 8, 128, 8192) == 0
    assert lib.gqa_decode_workspace_bytes(4, 32, 3, 128, 8192) == 0
    # the partials hold one fp32 row of d values + one log-sum-exp per split
    assert n >= 64 * 32 * 128 * 4


def test_decode_validation(lib):
    assert _decode(lib, q=None) == binding.GQA_ERR_NULL
    assert _decode(lib, lens=None) == binding.GQA_ERR_NULL
    assert _decode(lib, B=0) == binding.GQA_ERR_SHAPE
    assert _decode(lib, S_max=0) == binding.GQA_ERR_SHAPE
    assert _decode(lib, g=5) == binding.GQA_ERR_SHAPE
    assert _decode(lib, d=32) == binding.GQA_ERR_SHAPE
    assert _decode(lib, scale=-1.0) == binding.GQA_ERR_SHAPE
    assert _decode(lib, ws=None) == binding.GQA_ERR_WORKSPACE
    assert _decode(lib, ws_bytes=16) == binding.GQA_ERR_WORKSPACE
    assert _decode(lib, kc=MISALIGNED) == binding.GQA_ERR_ALIGN
    assert _decode(lib, ws=MISALIGNED) == binding.GQA_ERR_ALIGN
    assert _decode(lib, lens=FAKE + 2) == binding.GQA_ERR_ALIGN


def test_append_validation(lib):
    def app(kc=FAKE, vc=FAKE, lens=FAKE, kn=FAKE, vn=FAKE, B=2, g=2, d=64, S=16, T=1):
        return lib.kv_cache_append(kc, vc, lens, kn, vn, B, g, d, S, T, None, None)
    assert app(kc=None) == binding.GQA_ERR_NULL
    assert app(lens=None) == binding.GQA_ERR_NULL
    assert app(B=0) == binding.GQA_ERR_SHAPE
    assert app(d=48) == binding.GQA_ERR_SHAPE
    assert app(T=-1) == binding.GQA_ERR_SHAPE
    assert app(kn=MISALIGNED) == binding.GQA_ERR_ALIGN
    assert app(T=0) == binding.GQA_OK  # nothing to do, nothing queued


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        binding.load_library()


def test_variant_entry_points_validation(lib):
    f = FAKE

    def pre(causal=1, window=0, alibi=None, L=128):
        return lib.gqa_prefill_fwd_ex(f, f, f, f, 0, None, 1, L, 8, 2, 64, 0.125, causal, window,
                                      alibi, None, None)
    assert pre(window=-1) == binding.GQA_ERR_SHAPE
    assert pre(causal=0, window=16) == binding.GQA_ERR_SHAPE   # a window needs causal
    assert pre(alibi=FAKE + 2) == binding.GQA_ERR_ALIGN

    def cached(lens=f, T=16, S=1024, window=0):
        return lib.gqa_prefill_kvcache_fwd(f, f, f, lens, f, 0, None, 2, T, 32, 8, 128, S,
                                           0.088, window, None, None, None)
    assert cached(lens=None) == binding.GQA_ERR_NULL
    assert cached(T=2048, S=1024) == binding.GQA_ERR_SHAPE     # more new tokens than rows
    assert cached(T=0) == binding.GQA_ERR_SHAPE
    assert cached(window=-3) == binding.GQA_ERR_SHAPE
    assert cached(lens=FAKE + 2) == binding.GQA_ERR_ALIGN

    ws = lib.gqa_decode_workspace_bytes(4, 32, 8, 128, 1024)
    def dec(window=0, alibi=None):
        return lib.gqa_decode_fwd_ex(f, f, f, f, f, 0, None, 4, 32, 8, 128, 1024, 0.088, window,
                                     alibi, f, ws, None, None)
    assert dec(window=-1) == binding.GQA_ERR_SHAPE
    assert dec(alibi=FAKE + 1) == binding.GQA_ERR_ALIGN


def test_paged_entry_points_validation(lib):
    f = FAKE
    assert lib.gqa_decode_paged_workspace_bytes(4, 32, 8, 128, 16, 64) == \
        lib.gqa_decode_workspace_bytes(4, 32, 8, 128, 1024)
    assert lib.gqa_decode_paged_workspace_bytes(4, 32, 8, 128, 24, 64) == 0   # not a power of 2
    assert lib.gqa_decode_paged_workspace_bytes(4, 32, 8, 128, 8, 64) == 0    # page too small
    ws = lib.gqa_decode_paged_workspace_bytes(4, 32, 8, 128, 64, 16)

    def dec(table=f, page=64, pages=100, blocks=16):
        return lib.gqa_decode_paged_fwd(f, f, f, table, f, f, 0, None, 4, 32, 8, 128, page, pages,
                                        blocks, 0.088, 0, None, f, ws, None, None)
    assert dec(table=None) == binding.GQA_ERR_NULL
    assert dec(page=48) == binding.GQA_ERR_SHAPE
    assert dec(pages=0) == binding.GQA_ERR_SHAPE
    assert dec(table=FAKE + 2) == binding.GQA_ERR_ALIGN

    def app(table=f, page=64, T=1):
        return lib.kv_cache_append_paged(f, f, table, f, f, f, 2, 8, 128, page, 10, 4, T, None,
                                         None)
    assert app(table=None) == binding.GQA_ERR_NULL
    assert app(page=100) == binding.GQA_ERR_SHAPE
    assert app(T=0) == binding.GQA_OK


def test_rope_append_validation(lib):
    f = FAKE

    def app(q=f, q_out=f, cos=f, n_pos=4096, h_q=32, g=8, d=128, S=4096, T=1):
        # k_cache, v_cache, seq_lens, k_new, v_new, q, q_out, cos, sin, n_pos, B, h_q, g, d,
        # S_max, T, status, stream
        return lib.kv_cache_append_rope(f, f, f, f, f, q, q_out, cos, f, n_pos, 2, h_q, g, d, S,
                                        T, None, None)
    assert app(cos=None) == binding.GQA_ERR_NULL
    assert app(q_out=None) == binding.GQA_ERR_NULL          # q without q_out
    assert app(n_pos=4095) == binding.GQA_ERR_SHAPE          # a cache row without a table row
    assert app(h_q=12) == binding.GQA_ERR_SHAPE              # group size not a power of two
    assert app(d=96) == binding.GQA_ERR_SHAPE
    assert app(q_out=FAKE + 64) == binding.GQA_ERR_SHAPE     # q_out overlaps q partly
    assert app(cos=FAKE + 4) == binding.GQA_ERR_ALIGN
    assert app(T=0) == binding.GQA_OK                        # nothing to do, nothing queued
    assert app(q=None, q_out=None, T=0) == binding.GQA_OK

    def papp(table=f, page=64, blocks=16, n_pos=1024, T=1):
        return lib.kv_cache_append_paged_rope(f, f, table, f, f, f, f, f, f, f, n_pos, 2, 32, 8,
                                              128, page, 100, blocks, T, None, None)
    assert papp(table=None) == binding.GQA_ERR_NULL
    assert papp(page=48) == binding.GQA_ERR_SHAPE
    assert papp(n_pos=1023) == binding.GQA_ERR_SHAPE          # capacity 64 * 16 = 1024
    assert papp(T=0) == binding.GQA_OK


def test_selftest_bounded_wait_validation(lib):
    assert lib.gqa_selftest_bounded_wait(None, 1000, None) == binding.GQA_ERR_NULL
    assert lib.gqa_selftest_bounded_wait(FAKE, 0, None) == binding.GQA_ERR_SHAPE
    assert lib.gqa_selftest_bounded_wait(FAKE, 2000001, None) == binding.GQA_ERR_SHAPE
    assert lib.gqa_selftest_bounded_wait(FAKE + 2, 1000, None) == binding.GQA_ERR_ALIGN


def _expected_decode_workspace(B, h_q, g, d, S_max):
    """The decode workspace written out from the documented rule: split
    length = the fewest splits per segment (sequence, K/V head, 32-head slice)
    that give 80 % of the 296 CTA slots an item, in 64-token stages, capped at
    2048 tokens; four partials (O and log2 sum-exp) per split and query head,
    256-byte aligned sections, then a 16-byte counter."""
    slots, stage = 296, 64
    segs = B * g * ((h_q // g + 31) // 32)
    want = (slots * 4 + 4) // 5
    n = 1 if segs >= want else -(-want // segs)
    split = -(-S_max // n)
    split = min(2048, max(stage, -(-split // stage) * stage))
    n_split = -(-S_max // split)
    rows = B * h_q * n_split * 4
    lse_off = -(-(rows * d * 4) // 256) * 256
    counter_off = -(-(lse_off + rows * 4) // 256) * 256
    return counter_off + 16


@pytest.mark.parametrize("shape", [
    (32, 8, 4, 64, 1025),        # the bench step's decode
    (64, 32, 8, 128, 8192),      # ragged decode workload
    (16, 32, 1, 128, 32768),     # decode sweep g = 1
    (16, 32, 2, 128, 32768),     # decode sweep g = 2
    (16, 32, 32, 128, 32768),    # decode sweep g = 32
    (1, 8, 2, 64, 129),          # smoke
    (1, 128, 1, 64, 1),          # one row, G = 128 (four 32-head slices)
    (300, 64, 8, 128, 100000),   # many segments: one split per 2048 tokens
])
def test_decode_workspace_follows_the_split_rule(lib, shape):
    assert lib.gqa_decode_workspace_bytes(*shape) == _expected_decode_workspace(*shape)


C_CLIENT = r"""
#include <stdio.h>
#include "gqa.h"
int main(void) {
  /* host-only calls: no device needed */
  size_t ws = gqa_decode_workspace_bytes(64, 32, 8, 128, 8192);
  int rc_null = gqa_prefill_fwd(0, 0, 0, 0, GQA_OUT_F32, 0, 1, 128, 8, 2, 64, 0.125f, 1, 0, 0);
  int rc_shape = gqa_decode_fwd((void*)16, (void*)16, (void*)16, (const int*)16, (void*)16,
                                GQA_OUT_F32, 0, 2, 12, 8, 128, 1024, 0.1f, (void*)16, ws, 0, 0);
  printf("%d %zu %d %d %s\n", gqa_version(), ws, rc_null, rc_shape,
         gqa_status_string(GQA_ERR_CACHE_FULL));
  return 0;
}
"""


def test_plain_c_client_links_and_calls_the_library(tmp_path):
    """The boundary is a C ABI: a C99 program includes the header, links the
    shared library and gets the documented host-side answers."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    so = binding.LIB_PATH
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    str(src), so, f"-Wl,-rpath,{os.path.dirname(so)}", "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == binding.load_library().gqa_version()
    assert int(out[1]) == binding.load_library().gqa_decode_workspace_bytes(64, 32, 8, 128, 8192)
    assert int(out[2]) == binding.GQA_ERR_NULL      # null inputs
    assert int(out[3]) == binding.GQA_ERR_SHAPE     # h_q = 12 is not a multiple of g = 8
    assert out[4].startswith("GQA_ERR_CACHE_FULL")
