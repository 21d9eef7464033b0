"""Bucketed hash tables on the GPU (mp_build_buckets, mp_sampled_attention_buckets).

The build is checked against the oracle's bucket definition applied to the GPU's own codes:
offsets exactly, bucket contents as sets (their order is not fixed). The bucketed decode is
checked against the oracle's own bucket route ("LSH Sampling...", system co-design item 3: the
query's codes looked up in L tables; "don't pick the tallest", section 6): the oracle's tables of
the codes, each query's hits counted from its buckets, the sample sets exactly and the outputs
within 1e-3. It must also select exactly the keys the code scan selects.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import check_unit_buckets, row_rel_err
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


def _decode_check(mp, wl, x, W, centre, codes, buckets, units=None):
    """Bucketed decode (product call and its debug twin) against the oracle's bucket route on
    `units` (all by default); the scan's sample sets must be the same sets."""
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, *args),
                     dtype=torch.uint8, device="cuda")
    out_buck = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    mp.encode_query(x["q"], centre, W, x["keys"].shape, *args, ws)
    mp.sampled_attention_buckets(x["q"], buckets, centre, x["keys"], x["values"], *args,
                                 out_buck, ws)
    dbg = mp.debug_select_buckets(x["q"], buckets, codes, centre, W, x["keys"], x["values"],
                                  *args)
    scan = mp.debug_select(x["q"], codes, centre, W, x["keys"], x["values"], *args, counts=False)
    unpacked = mp.codes_unpack(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L) if wl.C else None
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    assert torch.equal(out_buck, dbg["out"])             # the debug twin runs the same kernels
    assert torch.equal(dbg["sel_count"], scan["sel_count"])
    assert torch.equal(dbg["sel_idx"], scan["sel_idx"])  # the same sets as the code scan
    gpu = {k: v.cpu().numpy() for k, v in dbg.items()}
    so = scan["out"].cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.Hq):
            assert row_rel_err(gpu["out"][b, h], so[b, h].astype(np.float64)) <= 1e-4
    xc = {k: v.cpu() for k, v in x.items()}
    up = unpacked.cpu().numpy() if unpacked is not None else None
    reps = []
    for b, g in units or [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]:
        reps.append(check_unit_buckets(b, g, q=xc["q"], keys=xc["keys"], values=xc["values"],
                                       centre=centre.cpu(), W=W.cpu(), K=wl.K, L=wl.L,
                                       n_sink=wl.n_sink, n_local=wl.n_local, gpu=gpu,
                                       unpacked=up))
    return reps


@pytest.mark.parametrize("shape", [
    dict(B=2, Hq=8, Hkv=2, n=5000, K=10, L=150, kv_dtype=BF),     # ragged last block, GQA 4
    dict(B=1, Hq=4, Hkv=4, n=3000, K=8, L=75, kv_dtype=F32),      # fp32, no GQA
    dict(B=1, Hq=8, Hkv=1, n=2048, K=12, L=20, kv_dtype=BF),      # the largest K, GQA 8
    dict(B=1, Hq=2, Hkv=1, n=1500, K=3, L=7, kv_dtype=BF),        # tiny tables: full buckets
    dict(B=1, Hq=4, Hkv=2, n=4100, K=9, L=40, kv_dtype=BF),       # 3 code words per transpose
    dict(B=1, Hq=4, Hkv=1, n=3333, K=11, L=30, kv_dtype=BF),      # 2 code words per transpose
])
def test_buckets_build_and_decode_against_the_oracle(mp, shape):
    wl = small_workload(**shape)
    x, W, centre, codes = _setup(mp, wl)
    buckets = _check_build(mp, wl, codes)
    reps = _decode_check(mp, wl, x, W, centre, codes, buckets)
    assert max(r.max_rel_err for r in reps) <= 1e-3


def test_buckets_degenerate_K0_and_single_table(mp):
    for K, L in ((0, 5), (6, 1)):
        wl = small_workload(B=1, Hq=4, Hkv=1, n=1100, K=K, L=L, kv_dtype=BF)
        x, W, centre, codes = _setup(mp, wl)
        buckets = mp.build_buckets(codes, wl.B, wl.Hkv, wl.n, K, L)
        reps = _decode_check(mp, wl, x, W, centre, codes, buckets)
        sizes = [s for r in reps for s in r.set_sizes]
        assert sizes == ([wl.n - wl.n_sink - wl.n_local] * wl.Hq if K == 0 else [0] * wl.Hq)


def test_buckets_long_context_three_kernel_build(mp):
    # ranges of 26+ blocks do not fit one CTA's shared memory: the counted three-kernel build
    wl = small_workload(B=1, Hq=2, Hkv=1, n=210_000, K=10, L=3, kv_dtype=BF)
    x, W, centre, codes = _setup(mp, wl)
    buckets = _check_build(mp, wl, codes)
    _decode_check(mp, wl, x, W, centre, codes, buckets)


def test_buckets_reject_too_many_bits(mp):
    assert mp.buckets_bytes(1, 1, 1000, 13, 10) == 0
    with pytest.raises(ValueError):
        mp.build_buckets(torch.zeros(16, dtype=torch.int32, device="cuda"), 1, 1, 1000, 13, 10)


def test_buckets_full_96k_layer_against_the_oracle(mp):
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
    # the full-size decode on the GPU; unit (0, 5) against the oracle's bucket route
    reps = _decode_check(mp, wl, x, W, centre, codes, buckets, units=[(0, 5)])
    assert reps[0].rows == wl.G and min(reps[0].set_sizes) > 0
