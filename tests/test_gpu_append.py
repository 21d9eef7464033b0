"""Caches laid out for more tokens than they hold, and the incremental append of decode tokens
(mp_key_mean_cap, mp_encode_keys, mp_build_buckets_cap, mp_params.n_capacity / n_indexed).

A cache with spare capacity must decode exactly like the same keys stored contiguously (the same
kernels run, only the strides change), so those outputs are compared bit for bit; the spare rows
hold large values that would show if anything read them. Appended keys are checked against the
oracle: after a prompt of n0 keys whose mean is the centre, keys are appended one at a time and
in chunks, and the decode at the final length is compared with the oracle's decode of all the
keys with the prompt's centre (sign bits inside the near-tie band are replayed as everywhere).
With bucketed tables built for the prompt, keys appended since come from the code scan of their
blocks, and that decode must select exactly what the scan selects.
"""
import pytest
import torch

from tests.parity import check_unit, check_unit_buckets
from workloads import make_hyperplanes, make_layer, small_workload

pytestmark = pytest.mark.gpu

BF, F32 = torch.bfloat16, torch.float32
SPARE = 100.0          # the value of every unused cache row


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_sampled_sparse_gb300 as mp
    mp.lib()
    return mp


def _cache(t, cap):
    """[B, Hkv, n, d] -> a [B, Hkv, cap, d] cache holding t in its first n rows."""
    B, Hkv, n, d = t.shape
    c = torch.full((B, Hkv, cap, d), SPARE, dtype=t.dtype, device="cuda")
    c[:, :, :n] = t.cuda()
    return c


def _codes(mp, wl, cap):
    return torch.empty(max(mp.codes_bytes(wl.B, wl.Hkv, cap, wl.K, wl.L) // 4, 4),
                       dtype=torch.int32, device="cuda")


def _decode_ws(mp, wl, n):
    return torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, n, wl.d, wl.K, wl.L,
                                                 wl.n_sink, wl.n_local),
                       dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("dt", [BF, F32])
def test_spare_capacity_decodes_like_the_contiguous_cache(mp, dt):
    wl = small_workload(B=2, Hq=8, Hkv=2, n=5000, kv_dtype=dt, q_dtype=dt, w_dtype=dt)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    centre = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], centre, W, wl.K, wl.L)
    want = mp.decode_attention(x["q"], codes, centre, W, x["keys"], x["values"], *args)

    cap = 7300
    kc, vc = _cache(x["keys"], cap), _cache(x["values"], cap)
    centre_c = mp.key_mean(kc, n=wl.n)
    codes_c = mp.encode_keys(kc, centre_c, W, wl.K, wl.L, 0, wl.n, _codes(mp, wl, cap))
    got = mp.decode_attention(x["q"], codes_c, centre_c, W, kc, vc, *args, n=wl.n)
    torch.cuda.synchronize()
    assert torch.equal(centre_c, centre)
    assert torch.equal(got, want)
    # the same codes, key by key (the capacity layout has more blocks per head)
    u = mp.codes_unpack(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    uc = mp.codes_unpack(codes_c, wl.B, wl.Hkv, cap, wl.K, wl.L)[:, :, :wl.n]
    assert torch.equal(u, uc)
    # the split halves and the bucketed tables on the capacity layout
    ws = _decode_ws(mp, wl, wl.n)
    out = torch.empty_like(want)
    mp.encode_query(x["q"], centre_c, W, kc.shape, *args, ws, n=wl.n)
    mp.sampled_attention(x["q"], codes_c, centre_c, kc, vc, *args, out, ws, n=wl.n)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    if dt == BF:
        # the bucketed decode on the capacity layout equals the one on the contiguous cache
        buckets = mp.build_buckets(codes_c, wl.B, wl.Hkv, wl.n, wl.K, wl.L, n_capacity=cap)
        mp.encode_query(x["q"], centre_c, W, kc.shape, *args, ws, n=wl.n)
        mp.sampled_attention_buckets(x["q"], buckets, centre_c, kc, vc, *args, out, ws, n=wl.n)
        b_contig = mp.build_buckets(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
        want_b = torch.empty_like(want)
        ws2 = _decode_ws(mp, wl, wl.n)
        mp.encode_query(x["q"], centre, W, x["keys"].shape, *args, ws2)
        mp.sampled_attention_buckets(x["q"], b_contig, centre, x["keys"], x["values"], *args,
                                     want_b, ws2)
        torch.cuda.synchronize()
        assert torch.equal(out, want_b)
    assert mp.device_status() == 0


def _append_case(mp, wl, n0, steps, cap):
    """Prompt of n0 keys, then the appends in `steps` ((begin, end) ranges); returns the cache,
    the prompt's centre and the codes."""
    x = make_layer(wl)
    W = make_hyperplanes(wl).cuda()
    kc, vc = _cache(x["keys"], cap), _cache(x["values"], cap)
    centre = mp.key_mean(kc, n=n0)
    codes = mp.encode_keys(kc, centre, W, wl.K, wl.L, 0, n0, _codes(mp, wl, cap))
    for a, b in steps:
        mp.encode_keys(kc, centre, W, wl.K, wl.L, a, b, codes)
    return x, W, kc, vc, centre, codes


def test_appended_keys_decode_like_the_oracle(mp):
    # prompt ends just before a word and block boundary (2048); single-key appends cross it, a
    # 40-key chunk takes the CUDA-core append, a 1000-key chunk re-encodes whole blocks
    wl = small_workload(B=1, Hq=4, Hkv=2, n=3100)
    n0, cap = 2030, 4096
    steps = [(i, i + 1) for i in range(n0, 2060)] + [(2060, 2100), (2100, 3100)]
    x, W, kc, vc, centre, codes = _append_case(mp, wl, n0, steps, cap)
    q = x["q"].cuda()
    dbg = mp.debug_select(q, codes, centre, W, kc, vc, wl.K, wl.L, wl.n_sink, wl.n_local,
                          n=wl.n)
    unpacked = mp.codes_unpack(codes, wl.B, wl.Hkv, cap, wl.K, wl.L)[:, :, :wl.n]
    torch.cuda.synchronize()
    gpu = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in dbg.items()}
    flips = 0
    for g in range(wl.Hkv):
        rep = check_unit(0, g, q=x["q"], keys=x["keys"], values=x["values"], centre=centre.cpu(),
                         W=W.cpu(), K=wl.K, L=wl.L, n_sink=wl.n_sink, n_local=wl.n_local,
                         gpu=gpu, unpacked=unpacked.cpu().numpy())
        flips += rep.key_flips
    assert flips <= 1e-5 * wl.Hkv * wl.n * wl.C
    assert mp.device_status() == 0


def test_fp32_appends_equal_a_full_build(mp):
    # fp32 keys and hyperplanes take the CUDA-core encoder for both the build and the appends,
    # with the same arithmetic, so the codes are identical bit for bit
    wl = small_workload(B=2, Hq=4, Hkv=2, n=2200, K=8, L=75, kv_dtype=F32, q_dtype=F32,
                        w_dtype=F32)
    n0, cap = 1000, 3000
    steps = [(i, i + 1) for i in range(n0, 1030)] + [(1030, 1094), (1094, 1100), (1100, 2200)]
    x, W, kc, vc, centre, codes = _append_case(mp, wl, n0, steps, cap)
    full = mp.build_tables(kc[:, :, :wl.n].contiguous(), centre, W, wl.K, wl.L)
    got = mp.codes_unpack(codes, wl.B, wl.Hkv, cap, wl.K, wl.L)[:, :, :wl.n]
    want = mp.codes_unpack(full, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    torch.cuda.synchronize()
    assert torch.equal(got, want)


@pytest.mark.parametrize("n0", [2500, 2048, 3100, 700])
def test_bucket_tables_plus_appended_tail_against_the_oracle(mp, n0):
    # tables built for the prompt (a ragged block, a block boundary, all keys, or less than one
    # block), keys appended since found by the scan of their blocks: the oracle's bucket route
    # over the first n0 keys plus direct counts for the scanned blocks gives the same sets
    wl = small_workload(B=2, Hq=8, Hkv=2, n=3100)
    cap = 4000
    steps = [(n0, wl.n)] if n0 < wl.n else []
    x, W, kc, vc, centre, codes = _append_case(mp, wl, n0, steps, cap)
    buckets = mp.build_buckets(codes, wl.B, wl.Hkv, n0, wl.K, wl.L, n_capacity=cap)
    q = x["q"].cuda()
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    ws = _decode_ws(mp, wl, wl.n)
    out_buck = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    mp.encode_query(q, centre, W, kc.shape, *args, ws, n=wl.n)
    mp.sampled_attention_buckets(q, buckets, centre, kc, vc, *args, out_buck, ws, codes=codes,
                                 n=wl.n, n_indexed=n0)
    dbg = mp.debug_select_buckets(q, buckets, codes, centre, W, kc, vc, *args, n=wl.n,
                                  n_indexed=n0)
    scan = mp.debug_select(q, codes, centre, W, kc, vc, *args, n=wl.n, counts=False)
    unpacked = mp.codes_unpack(codes, wl.B, wl.Hkv, cap, wl.K, wl.L)[:, :, :wl.n]
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    assert torch.equal(out_buck, dbg["out"])
    assert torch.equal(dbg["sel_idx"], scan["sel_idx"])
    gpu = {k: v.cpu().numpy() for k, v in dbg.items()}
    for b in range(wl.B):
        for g in range(wl.Hkv):
            check_unit_buckets(b, g, q=x["q"], keys=x["keys"], values=x["values"],
                               centre=centre.cpu(), W=W.cpu(), K=wl.K, L=wl.L, n_sink=wl.n_sink,
                               n_local=wl.n_local, gpu=gpu, unpacked=unpacked.cpu().numpy(),
                               n_indexed=n0)
