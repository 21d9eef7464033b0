"""The MIPS -> cosine variant on the GPU (mp_key_radius, mp_encode_keys_mips, MP_FLAG_MIPS).

Keys are centred and extended by sqrt(r^2 - |k - mu|^2), r the longest centred key; W has a
(d + 1)-th row for that coordinate and the query uses the first d rows. The radius is compared
with the oracle's fp64 value, then passed to the oracle as the GPU used it (like the centre); the
codes, sample sets and outputs are compared with the oracle's MIPS decode under the usual
near-tie replay of sign bits.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import check_unit, row_rel_err
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


def _w_aug(wl):
    """[d + 1, K*L] hyperplanes, seeded like the workload's own."""
    return make_hyperplanes(wl.replace(d=wl.d + 1)).contiguous()


@pytest.mark.parametrize("shape,tensor_cores", [
    (dict(B=1, Hq=4, Hkv=2, n=3000, K=10, L=150, kv_dtype=BF), True),
    (dict(B=1, Hq=4, Hkv=2, n=3000, K=10, L=150, kv_dtype=BF), False),
    (dict(B=2, Hq=2, Hkv=1, n=1500, K=8, L=75, kv_dtype=F32, q_dtype=F32, w_dtype=F32), True),
    # 20 blocks per head, the last of 544 keys: each encoder CTA takes several units, so the key
    # slices' norms are fetched ahead across blocks, ragged blocks and heads
    (dict(B=2, Hq=8, Hkv=4, n=20000, K=10, L=150, kv_dtype=BF), True),
])
def test_mips_decode_matches_the_oracle(mp, shape, tensor_cores):
    # bf16 with tensor_cores: the tcgen05 encoder takes the extra coordinate into its first MMA
    # step (per-tile key slices beside the centre)
    wl = small_workload(**shape)
    x = make_layer(wl)
    xc = {k: v.cuda() for k, v in x.items()}
    W = _w_aug(wl)
    Wc = W.cuda()
    centre = mp.key_mean(xc["keys"])
    radius = mp.key_radius(xc["keys"], centre)
    codes = mp.encode_keys_mips(xc["keys"], centre, Wc, radius, wl.K, wl.L, 0, wl.n,
                                tensor_cores=tensor_cores)
    dbg = mp.debug_select(xc["q"], codes, centre, Wc, xc["keys"], xc["values"], wl.K, wl.L,
                          wl.n_sink, wl.n_local, radius=radius)
    prod = mp.decode_attention(xc["q"], codes, centre, Wc, xc["keys"], xc["values"], wl.K, wl.L,
                               wl.n_sink, wl.n_local, radius=radius)
    unpacked = mp.codes_unpack(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    assert torch.equal(prod, dbg["out"])
    gpu = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in dbg.items()}
    rad = radius.cpu().double().numpy()
    cen = centre.cpu()
    flips = 0
    for b in range(wl.B):
        for g in range(wl.Hkv):
            want = O.mips_radius(x["keys"][b, g], cen[b, g])
            assert abs(rad[b, g] - want) <= 1e-5 * want
            rep = check_unit(b, g, q=x["q"], keys=x["keys"], values=x["values"], centre=cen, W=W,
                             K=wl.K, L=wl.L, n_sink=wl.n_sink, n_local=wl.n_local, gpu=gpu,
                             unpacked=unpacked.cpu().numpy(), radius=rad[b, g])
            flips += rep.key_flips
            assert all(s > 0 for s in rep.set_sizes)
    assert flips <= 1e-5 * wl.B * wl.Hkv * wl.n * wl.C


def test_mips_ranges_equal_a_full_encode_and_buckets_select_like_the_scan(mp):
    wl = small_workload(B=2, Hq=8, Hkv=2, n=2600)
    xc = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = _w_aug(wl).cuda()
    centre = mp.key_mean(xc["keys"])
    radius = mp.key_radius(xc["keys"], centre)
    # the CUDA-core encoder over ranges gives the codes of one pass over all keys, bit for bit
    full = mp.encode_keys_mips(xc["keys"], centre, W, radius, wl.K, wl.L, 0, wl.n,
                               tensor_cores=False)
    parts = torch.zeros_like(full)
    for a, b in [(0, 1000), (1000, 1001), (1001, 1030), (1030, 2047), (2047, 2600)]:
        mp.encode_keys_mips(xc["keys"], centre, W, radius, wl.K, wl.L, a, b, parts,
                            tensor_cores=False)
    u_full = mp.codes_unpack(full, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    u_parts = mp.codes_unpack(parts, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    assert torch.equal(u_full, u_parts)
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, *args),
                     dtype=torch.uint8, device="cuda")
    out_scan = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    out_buck = torch.empty_like(out_scan)
    mp.encode_query(xc["q"], centre, W, xc["keys"].shape, *args, ws, radius=radius)
    mp.sampled_attention(xc["q"], full, centre, xc["keys"], xc["values"], *args, out_scan, ws,
                         radius=radius)
    buckets = mp.build_buckets(full, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    mp.encode_query(xc["q"], centre, W, xc["keys"].shape, *args, ws, radius=radius)
    mp.sampled_attention_buckets(xc["q"], buckets, centre, xc["keys"], xc["values"], *args,
                                 out_buck, ws, radius=radius)
    # the two retrievals select the same sets; the gathers of those sets agree to rounding
    sel_s = mp.debug_select(xc["q"], full, centre, W, xc["keys"], xc["values"], *args,
                            counts=False, radius=radius)
    sel_b = mp.debug_select_buckets(xc["q"], buckets, full, centre, W, xc["keys"], xc["values"],
                                    *args, radius=radius)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    assert torch.equal(sel_s["sel_idx"], sel_b["sel_idx"])
    assert torch.equal(out_buck, sel_b["out"]) and torch.equal(out_scan, sel_s["out"])
    gs, gb = out_scan.cpu().numpy(), out_buck.cpu().numpy()
    for b in range(wl.B):
        for h in range(wl.Hq):
            assert row_rel_err(gb[b, h], gs[b, h].astype(np.float64)) <= 1e-4
    # the variant samples differently from the plain cosine on the same keys
    plain = mp.decode_attention(xc["q"], mp.build_tables(xc["keys"], centre, W[:wl.d].contiguous(),
                                                         wl.K, wl.L),
                                centre, W[:wl.d].contiguous(), xc["keys"], xc["values"], *args)
    assert not torch.equal(plain, out_scan)
    assert np.isfinite(out_scan.cpu().numpy()).all()


def test_mips_full_96k_layer_against_the_oracle(mp):
    # one layer of the 96K workload (B=1, 32 query heads over 8 KV heads, n = 98,304) encoded on
    # the tensor cores as the bench does; two (sequence, KV head) units checked against the oracle
    wl = WORKLOADS["llama8b_n96k_32layers"]
    x = make_layer(wl, 0)
    xc = {k: v.cuda() for k, v in x.items()}
    W = _w_aug(wl)
    Wc = W.cuda()
    centre = mp.key_mean(xc["keys"])
    radius = mp.key_radius(xc["keys"], centre)
    codes = mp.encode_keys_mips(xc["keys"], centre, Wc, radius, wl.K, wl.L, 0, wl.n)
    dbg = mp.debug_select(xc["q"], codes, centre, Wc, xc["keys"], xc["values"], wl.K, wl.L,
                          wl.n_sink, wl.n_local, counts=False, radius=radius)
    unpacked = mp.codes_unpack(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L).cpu().numpy()
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    gpu = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in dbg.items()}
    rad = radius.cpu().double().numpy()
    cen = centre.cpu()
    flips = 0
    for b, g in [(0, 0), (0, 5)]:
        want = O.mips_radius(x["keys"][b, g], cen[b, g])
        assert abs(rad[b, g] - want) <= 1e-5 * want
        rep = check_unit(b, g, q=x["q"], keys=x["keys"], values=x["values"], centre=cen, W=W,
                         K=wl.K, L=wl.L, n_sink=wl.n_sink, n_local=wl.n_local, gpu=gpu,
                         unpacked=unpacked, radius=rad[b, g], check_counts=False)
        flips += rep.key_flips
        assert rep.rows == wl.G and all(sz > 0 for sz in rep.set_sizes)
    assert flips <= 1e-5 * 2 * wl.n * wl.C
