"""Bucketed hash tables on the GPU (mp_build_buckets, mp_sampled_attention_buckets).

The build is checked against the oracle's bucket definition applied to the GPU's own codes:
offsets exactly, bucket contents as sets (their order is not fixed). The bucketed decode must
select exactly the keys the code scan selects, so its output equals the scan's output bit for
bit on the same inputs (the gather, weights and merge are the same kernel); the scan's own parity
with the oracle is covered in test_gpu_parity.py.
"""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import WORKLOADS, make_hyperplanes, make_layer, small_workload

pytestmark = pytest.mark.gpu

BF, F32 = torch.bfloat16, torch.float32


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_sampled_sparse_gb300 as mp
    mp.lib()
    return mp


def _setup(mp, wl, layer=0):
    x = {k: v.cuda() for k, v in make_layer(wl, layer).items()}
    W = make_hyperplanes(wl).cuda()
    ws = torch.empty(max(mp.key_mean_workspace_bytes(wl.B, wl.Hkv, wl.n, wl.d), 256),
                     dtype=torch.uint8, device="cuda")
    centre = mp.key_mean(x["keys"], workspace=ws)
    codes = mp.build_tables(x["keys"], centre, W, wl.K, wl.L)
    return x, W, centre, codes


def _unpack_buckets(buckets, B, Hkv, n, K, L):
    nb = 1 << K
    per = L * (nb + 1 + n + 8 * nb)               # offsets, members, build scratch
    flat = buckets.cpu().numpy().astype(np.int64)[:B * Hkv * per].reshape(B * Hkv, per)
    offsets = flat[:, :L * (nb + 1)].reshape(B * Hkv, L, nb + 1)
    members = flat[:, L * (nb + 1):L * (nb + 1 + n)].reshape(B * Hkv, L, n)
    return offsets, members


def _check_build(mp, wl, codes):
    B, Hkv, n, K, L = wl.B, wl.Hkv, wl.n, wl.K, wl.L
    buckets = mp.build_buckets(codes, B, Hkv, n, K, L)
    torch.cuda.synchronize()
    got_off, got_mem = _unpack_buckets(buckets, B, Hkv, n, K, L)
    gpu_codes = mp.codes_unpack(codes, B, Hkv, n, K, L).cpu().numpy()   # the GPU's own codes
    for bg in range(B * Hkv):
        want_off, want_mem = O.bucket_tables(gpu_codes[bg // Hkv, bg % Hkv], K, L)
        assert np.array_equal(got_off[bg], want_off), f"offsets differ in unit {bg}"
        for t in range(L):
            for c in np.nonzero(np.diff(want_off[t]))[0]:
                lo, hi = want_off[t, c], want_off[t, c + 1]
                assert np.array_equal(np.sort(got_mem[bg, t, lo:hi]), want_mem[t, lo:hi]), \
                    f"bucket {c} of table {t} differs in unit {bg}"
    return buckets


def _decode_both(mp, wl, x, W, centre, codes, buckets):
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, wl.K, wl.L,
                                               wl.n_sink, wl.n_local),
                     dtype=torch.uint8, device="cuda")
    out_scan = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    out_buck = torch.empty_like(out_scan)
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    mp.encode_query(x["q"], centre, W, x["keys"].shape, *args, ws)
    mp.sampled_attention(x["q"], codes, centre, x["keys"], x["values"], *args, out_scan, ws)
    mp.encode_query(x["q"], centre, W, x["keys"].shape, *args, ws)
    mp.sampled_attention_buckets(x["q"], buckets, centre, x["keys"], x["values"], *args,
                                 out_buck, ws)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    return out_scan.cpu().numpy(), out_buck.cpu().numpy()


@pytest.mark.parametrize("shape", [
    dict(B=2, Hq=8, Hkv=2, n=5000, K=10, L=150, kv_dtype=BF),     # ragged last block, GQA 4
    dict(B=1, Hq=4, Hkv=4, n=3000, K=8, L=75, kv_dtype=F32),      # fp32, no GQA
    dict(B=1, Hq=8, Hkv=1, n=2048, K=12, L=20, kv_dtype=BF),      # the largest K, GQA 8
    dict(B=1, Hq=2, Hkv=1, n=1500, K=3, L=7, kv_dtype=BF),        # tiny tables: full buckets
    dict(B=1, Hq=4, Hkv=2, n=4100, K=9, L=40, kv_dtype=BF),       # 3 code words per transpose
    dict(B=1, Hq=4, Hkv=1, n=3333, K=11, L=30, kv_dtype=BF),      # 2 code words per transpose
])
def test_buckets_build_and_decode_match_the_scan(mp, shape):
    wl = small_workload(**shape)
    x, W, centre, codes = _setup(mp, wl)
    buckets = _check_build(mp, wl, codes)
    out_scan, out_buck = _decode_both(mp, wl, x, W, centre, codes, buckets)
    assert np.array_equal(out_scan, out_buck)


def test_buckets_degenerate_K0_and_single_table(mp):
    for K, L in ((0, 5), (6, 1)):
        wl = small_workload(B=1, Hq=4, Hkv=1, n=1100, K=K, L=L, kv_dtype=BF)
        x, W, centre, codes = _setup(mp, wl)
        buckets = mp.build_buckets(codes, wl.B, wl.Hkv, wl.n, K, L)
        out_scan, out_buck = _decode_both(mp, wl, x, W, centre, codes, buckets)
        assert np.array_equal(out_scan, out_buck)


def test_buckets_long_context_three_kernel_build(mp):
    # ranges of 26+ blocks do not fit one CTA's shared memory: the counted three-kernel build
    wl = small_workload(B=1, Hq=2, Hkv=1, n=210_000, K=10, L=3, kv_dtype=BF)
    x, W, centre, codes = _setup(mp, wl)
    buckets = _check_build(mp, wl, codes)
    out_scan, out_buck = _decode_both(mp, wl, x, W, centre, codes, buckets)
    assert np.array_equal(out_scan, out_buck)


def test_buckets_reject_too_many_bits(mp):
    assert mp.buckets_bytes(1, 1, 1000, 13, 10) == 0
    with pytest.raises(ValueError):
        mp.build_buckets(torch.zeros(16, dtype=torch.int32, device="cuda"), 1, 1, 1000, 13, 10)


def test_buckets_full_96k_layer_matches_the_scan(mp):
    wl = WORKLOADS["llama8b_n96k_32layers"]
    x, W, centre, codes = _setup(mp, wl, layer=3)
    buckets = mp.build_buckets(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    # one unit's tables in full against the definition
    gpu_codes = mp.codes_unpack(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)[0, 5].cpu().numpy()
    off, mem = _unpack_buckets(buckets, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    want_off, want_mem = O.bucket_tables(gpu_codes, wl.K, wl.L)
    assert np.array_equal(off[5], want_off)
    for t in (0, 77, wl.L - 1):
        got = np.concatenate([np.sort(mem[5, t, want_off[t, c]:want_off[t, c + 1]])
                              for c in range(1 << wl.K)])
        assert np.array_equal(got, want_mem[t])
    out_scan, out_buck = _decode_both(mp, wl, x, W, centre, codes, buckets)
    assert np.array_equal(out_scan, out_buck)
