"""The C ABI on the host, with no GPU work: the library loads, exports what the header declares,
and rejects bad arguments before anything could be launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "magicpig.h")


@pytest.fixture(scope="module")
def L():
    from lsh_sampled_sparse_gb300.build import build
    build()
    import lsh_sampled_sparse_gb300 as mp
    return mp.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^MP_API\s+[\w\s\*]+?\b(mp_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("mp_key_mean", "mp_build_tables", "mp_decode_attention", "mp_encode_query",
                 "mp_sampled_attention", "mp_debug_select", "mp_codes_unpack",
                 "mp_device_status", "mp_codes_bytes"):
        assert must in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings_and_version(L):
    import lsh_sampled_sparse_gb300 as mp
    header_version = int(re.search(r"#define MP_ABI_VERSION (\d+)", open(HEADER).read()).group(1))
    assert mp.abi_version() == header_version
    assert ctypes.sizeof(mp.Params) == 48          # mp_params: 8 four-byte fields, 2 pointers
    names = [L.mp_status_string(i).decode() for i in range(7)]
    assert names == ["MP_OK", "MP_ERR_INVALID_ARG", "MP_ERR_UNSUPPORTED", "MP_ERR_CUDA",
                     "MP_ERR_TIMEOUT", "MP_ERR_WORKSPACE", "MP_ERR_BOUNDS"]


def test_codes_bytes(L):
    import lsh_sampled_sparse_gb300 as mp
    # 1024-key blocks of K*L rows of 128 bytes: 187.5 bytes per key at (10, 150)
    assert mp.codes_bytes(1, 8, 98304, 10, 150) == 8 * 96 * 1500 * 128
    assert mp.codes_bytes(1, 1, 98304, 10, 150) / 98304 == 187.5
    assert mp.codes_bytes(1, 1, 1, 10, 150) == 1500 * 128          # padded to a block
    assert mp.codes_bytes(2, 3, 1025, 8, 75) == 2 * 3 * 2 * 600 * 128
    assert mp.codes_bytes(1, 1, 100, 0, 4) == 0
    assert mp.codes_bytes(0, 1, 100, 10, 150) == 0


def test_workspace_sizes(L):
    import lsh_sampled_sparse_gb300 as mp
    assert mp.decode_workspace_bytes(1, 32, 8, 98304, 128, 10, 150, 4, 64) > 0
    assert mp.debug_workspace_bytes(1, 32, 8, 98304, 128, 10, 150, 4, 64) >= \
        mp.decode_workspace_bytes(1, 32, 8, 98304, 128, 10, 150, 4, 64)
    assert mp.decode_workspace_bytes(1, 32, 7, 1000, 128, 10, 150, 4, 64) == 0   # Hq % Hkv
    assert mp.decode_workspace_bytes(1, 4, 1, 1000, 128, 33, 2, 4, 64) == 0      # K > 32
    assert mp.decode_workspace_bytes(1, 4, 1, 1000, 128, 10, 0, 4, 64) == 0      # L < 1
    assert mp.decode_workspace_bytes(1, 4, 1, 1000, 128, 10, 5, -1, 64) == 0     # n_sink < 0
    assert mp.key_mean_workspace_bytes(1, 8, 98304, 128) > 0
    assert mp.key_mean_workspace_bytes(1, 8, 98304, 64) == 0


@pytest.mark.parametrize("B,Hkv,n,rows", [
    (1, 8, 98304, 1024),     # 96 ranges per head x 8 heads = 768: long ranges
    (4, 8, 16384, 512),      # 16 x 32 = 512 < 608 ranges: halved once
    (1, 1, 4096, 64),        # a single short head: the 64-key floor
    (32, 8, 32768, 1024),    # many heads: long ranges
    (1, 1, 100, 64),         # one short range
])
def test_key_mean_ranges_fill_the_gpu(B, Hkv, n, rows):
    # the workspace holds one 128-float range sum per (head, range) plus a counter per head;
    # ranges are 1024 keys, halved down to 64 while the heads would have fewer than 608 of them
    import lsh_sampled_sparse_gb300 as mp
    ranges = (n + rows - 1) // rows
    want = B * Hkv * ranges * 128 * 4 + B * Hkv * 4
    assert mp.key_mean_workspace_bytes(B, Hkv, n, 128) == (want + 255) // 256 * 256


def _decode(L, ws_bytes=1 << 20, d=128, Hq=4, Hkv=1, n=1000, K=10, Lt=150, flags=0,
            null_q=False, ptr=0x10000):
    import lsh_sampled_sparse_gb300 as mp
    p = mp.Params(K, Lt, 4, 64, 0.0, flags)
    P = ctypes.c_void_p
    q = None if null_q else P(ptr)
    return L.mp_decode_attention(q, 1, P(ptr), P(ptr), P(ptr), 1, P(ptr), P(ptr), 1, 1, Hq, Hkv,
                                 n, d, ctypes.byref(p), P(ptr), P(ptr), ws_bytes, None)


def test_decode_rejects_bad_arguments_before_launch(L):
    INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 5
    assert _decode(L, null_q=True) == INVALID
    assert _decode(L, Hq=6, Hkv=4) == INVALID
    assert _decode(L, flags=1) == INVALID
    assert _decode(L, K=-1) == INVALID
    assert _decode(L, ptr=0x10004) == INVALID                   # misaligned pointers
    assert _decode(L, d=64) == UNSUPPORTED
    assert _decode(L, Hq=3, Hkv=1) == UNSUPPORTED               # GQA group of 3
    assert _decode(L, Hq=16, Hkv=1) == UNSUPPORTED              # GQA group of 16
    assert _decode(L, ws_bytes=16) == WORKSPACE


def test_split_halves_reject_bad_arguments_before_launch(L):
    import lsh_sampled_sparse_gb300 as mp
    P = ctypes.c_void_p
    ok = P(0x10000)
    p = mp.Params(10, 150, 4, 64, 0.0, 0)
    assert L.mp_encode_query(None, 1, ok, ok, 1, 1, 4, 1, 1000, 128, ctypes.byref(p), ok,
                             1 << 20, None) == 1
    assert L.mp_encode_query(ok, 1, ok, ok, 1, 1, 4, 1, 1000, 64, ctypes.byref(p), ok,
                             1 << 20, None) == 2
    assert L.mp_encode_query(ok, 1, ok, ok, 1, 1, 4, 1, 1000, 128, ctypes.byref(p), ok,
                             16, None) == 5
    assert L.mp_sampled_attention(ok, 1, None, ok, ok, ok, 1, 1, 4, 1, 1000, 128,
                                  ctypes.byref(p), ok, ok, 1 << 20, None) == 1
    assert L.mp_sampled_attention(ok, 1, ok, ok, ok, ok, 1, 1, 4, 1, 1000, 128,
                                  ctypes.byref(p), ok, ok, 16, None) == 5


def test_build_and_mean_reject_bad_arguments(L):
    P = ctypes.c_void_p
    ok = P(0x10000)
    assert L.mp_build_tables(None, 1, ok, ok, 1, 1, 1, 100, 128, 10, 150, ok, None) == 1
    assert L.mp_build_tables(ok, 1, ok, ok, 1, 1, 1, 100, 64, 10, 150, ok, None) == 2
    assert L.mp_build_tables(ok, 1, ok, ok, 1, 1, 1, 100, 128, 33, 150, ok, None) == 1
    assert L.mp_build_tables(ok, 7, ok, ok, 1, 1, 1, 100, 128, 10, 150, ok, None) == 1
    assert L.mp_build_tables(P(0x10002), 1, ok, ok, 1, 1, 1, 100, 128, 10, 150, ok, None) == 1
    # K == 0: nothing to encode, nothing touched
    assert L.mp_build_tables(None, 1, None, None, 1, 1, 1, 100, 128, 0, 150, None, None) == 0
    assert L.mp_key_mean(ok, 1, 1, 1, 0, 128, ok, ok, 1 << 20, None) == 1
    assert L.mp_key_mean(ok, 1, 1, 1, 100, 64, ok, ok, 1 << 20, None) == 2
    assert L.mp_key_mean(ok, 1, 1, 8, 98304, 128, ok, ok, 16, None) == 5


def test_capacity_and_append_reject_bad_arguments(L):
    import lsh_sampled_sparse_gb300 as mp
    P = ctypes.c_void_p
    ok = P(0x10000)
    INVALID = 1

    def ws(n, n_capacity=0, n_indexed=0):
        p = mp.Params(10, 150, 4, 64, 0.0, 0, n_capacity, n_indexed)
        return L.mp_decode_workspace_bytes(1, 4, 1, n, 128, ctypes.byref(p))
    assert ws(1000) > 0 and ws(1000, 4096) == ws(1000) and ws(1000, 0, 500) == ws(1000)
    assert ws(1000, 999) == 0                     # capacity below the length
    assert ws(1000, -1) == 0
    assert ws(1000, 0, 1001) == 0                 # more keys indexed than cached
    # mp_encode_keys(keys, dt, centre, W, wdt, B, Hkv, n_capacity, n_begin, n_end, d, K, L, codes)
    def enc(cap, n0, n1, d=128, K=10, keys=ok):
        return L.mp_encode_keys(keys, 1, ok, ok, 1, 1, 1, cap, n0, n1, d, K, 150, ok, None)
    assert enc(4096, 100, 4097) == INVALID        # past the capacity
    assert enc(4096, -1, 10) == INVALID
    assert enc(4096, 20, 10) == INVALID           # reversed range
    assert enc(4096, 0, 10, d=64) == 2
    assert enc(4096, 0, 10, keys=None) == INVALID
    assert enc(4096, 10, 10, keys=None) == 0      # empty range: nothing touched
    assert enc(4096, 0, 10, K=0, keys=None) == 0  # no hyperplanes
    assert L.mp_key_mean_cap(ok, 1, 1, 1, 99, 100, 128, ok, ok, 1 << 20, None) == INVALID
    assert L.mp_build_buckets_cap(ok, 1, 1, 99, 100, 10, 150, ok, None) == INVALID
    # the bucketed decode needs the codes for keys appended after the tables were built
    p = mp.Params(10, 150, 4, 64, 0.0, 0, 0, 500)
    assert L.mp_sampled_attention_buckets(ok, 1, ok, None, ok, ok, ok, 1, 1, 4, 1, 1000, 128,
                                          ctypes.byref(p), ok, ok, 1 << 24, None) == INVALID


def test_mips_variant_rejects_bad_arguments(L):
    import lsh_sampled_sparse_gb300 as mp
    P = ctypes.c_void_p
    ok = P(0x10000)

    def ws(flags, radius):
        p = mp.Params(10, 150, 4, 64, 0.0, flags, 0, 0, radius)
        return L.mp_decode_workspace_bytes(1, 4, 1, 1000, 128, ctypes.byref(p))
    assert ws(0, None) > 0 and ws(mp.MP_FLAG_MIPS, 0x10000) == ws(0, None)
    assert ws(mp.MP_FLAG_MIPS, None) == 0        # the variant needs its radii
    assert ws(0, 0x10000) == 0                   # radii without the flag
    assert ws(2, None) == 0                      # unknown flag
    assert ws(mp.MP_FLAG_MIPS, 0x10002) == 0     # misaligned radii
    # mp_key_radius(keys, dt, centre, B, Hkv, n_capacity, n, d, radius)
    assert L.mp_key_radius(ok, 1, ok, 1, 1, 100, 100, 128, None, None) == 1
    assert L.mp_key_radius(ok, 1, ok, 1, 1, 99, 100, 128, ok, None) == 1
    assert L.mp_key_radius(ok, 1, ok, 1, 1, 100, 100, 64, ok, None) == 2
    # mp_encode_keys_mips(keys, dt, centre, W, wdt, radius, B, Hkv, cap, n0, n1, d, K, L, codes)
    assert L.mp_encode_keys_mips(ok, 1, ok, ok, 1, None, 1, 1, 100, 0, 100, 128, 10, 150, ok,
                                 None, None) == 1
    assert L.mp_encode_keys_mips(ok, 1, ok, ok, 1, ok, 1, 1, 100, 0, 101, 128, 10, 150, ok,
                                 None, None) == 1
    assert L.mp_encode_keys_mips(ok, 1, ok, ok, 1, ok, 1, 1, 100, 0, 100, 128, 10, 150, ok,
                                 P(0x10002), None) == 1          # misaligned scratch
    assert L.mp_encode_keys_mips(None, 1, None, None, 1, None, 1, 1, 100, 5, 5, 128, 10, 150,
                                 None, None, None) == 0


def test_cross_polytope_variant_rejects_bad_arguments(L):
    import lsh_sampled_sparse_gb300 as mp
    P = ctypes.c_void_p
    ok = P(0x10000)
    CP, MIPS = mp.MP_FLAG_CROSS_POLYTOPE, mp.MP_FLAG_MIPS

    def ws(K, flags, radius=None, table=None):
        p = mp.Params(K, 20, 4, 64, 0.0, flags, 0, 0, radius, table)
        return L.mp_decode_workspace_bytes(1, 4, 1, 1000, 128, ctypes.byref(p))
    assert ws(1, CP, table=0x10000) > 0
    assert ws(1, CP) == 0                         # the variant needs its log u table
    assert ws(2, CP, table=0x10000) == 0          # one hash per table
    assert ws(1, CP | MIPS, 0x10000, 0x10000) == 0
    assert ws(1, 0, table=0x10000) == 0           # a table without the flag
    assert ws(1, CP, table=0x10002) == 0          # misaligned table
    assert L.mp_cp_logu_table(0, 20, 128, ok, None) == 1
    assert L.mp_cp_logu_table(1, 20, 64, ok, None) == 2
    assert L.mp_cp_logu_table(1, 20, 128, None, None) == 1
    assert L.mp_cp_codes_bytes(1, 8, 98304, 20) == 8 * 96 * 20 * 1024
    assert L.mp_cp_codes_bytes(1, 8, 0, 20) == 0
    # mp_encode_keys_cp(keys, dt, centre, G, gdt, B, Hkv, cap, n0, n1, d, L, codes)
    assert L.mp_encode_keys_cp(ok, 1, ok, ok, 1, 1, 1, 100, 0, 101, 128, 20, ok, None) == 1
    assert L.mp_encode_keys_cp(ok, 1, ok, ok, 1, 1, 1, 100, 0, 50, 64, 20, ok, None) == 2
    assert L.mp_encode_keys_cp(None, 1, None, None, 1, 1, 1, 100, 7, 7, 128, 20, None,
                               None) == 0


def test_binding_refuses_cpu_tensors(L):
    import torch

    import lsh_sampled_sparse_gb300 as mp
    with pytest.raises(TypeError):
        mp.key_mean(torch.zeros(1, 1, 16, 128))


def test_package_has_no_cpu_fallback_and_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "lsh_sampled_sparse_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_checks_build_compiles_and_exports_the_same_symbols():
    # the MP_CHECKS build (index checks that raise MP_ERR_BOUNDS) is the same boundary
    from lsh_sampled_sparse_gb300.build import build
    path = build(checks=True)
    assert path.endswith("libmagicpig_checks.so")
    C = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(C, n)]
    assert not missing, missing
    C.mp_status_string.restype = ctypes.c_char_p
    assert C.mp_status_string(6) == b"MP_ERR_BOUNDS"
