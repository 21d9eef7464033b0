"""The cross-polytope variant on the GPU (mp_cp_logu_table, mp_encode_keys_cp,
MP_FLAG_CROSS_POLYTOPE).

Table t hashes to the signed argmax of |G_t x| (G_t Gaussian, d x d), one byte; one hash per
table. The GPU's log u table is compared with the oracle's quadrature; codes, sample sets and
outputs with the oracle's decode, where a code may differ only at a near tie of the two largest
coordinates and must then be the runner-up (replayed into the oracle, as sign bits are for
SimHash).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import OUT_REL_TOL, row_rel_err
from workloads import WORKLOADS, make_layer, small_workload

pytestmark = pytest.mark.gpu

BF, F32 = torch.bfloat16, torch.float32
L_CP = 16


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_sampled_sparse_gb300 as mp
    mp.lib()
    return mp


def _rotations(L, d, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(L, d, d, generator=g).to(dtype).contiguous()


def _unpack(codes, B, Hkv, n, L):
    """bytes [B*Hkv][blocks][L][1024] -> [B, Hkv, n, L]"""
    nblk = (n + 1023) // 1024
    c = codes.cpu().numpy().reshape(B, Hkv, nblk, L, 1024)
    return np.transpose(c, (0, 1, 2, 4, 3)).reshape(B, Hkv, nblk * 1024, L)[:, :, :n].astype(np.int64)


def test_cp_logu_table_matches_the_oracle(mp):
    K, L = 1, L_CP
    table = mp.cp_logu_table(K, L).cpu().double().numpy()
    assert table.shape == (4097,)
    idx = np.array([0, 205, 410, 820, 1228, 1638, 2048, 2458, 2867, 3277, 3686, 3993, 4010,
                    4050, 4075, 4090, 4096])
    c = np.minimum(1.0, -1.0 + 2.0 * idx / 4096)
    p = O.cp_collision_probability(c, 128)
    want = O.log_inclusion_probability(p, K, L)
    for i, w, g in zip(idx, want, table[idx]):
        if not np.isfinite(w) or w < -87.0:            # p = 0: fp32 clamps to log(FLT_MIN)
            assert g <= -87.0
        else:
            assert abs(g - w) <= 2e-4 * max(1.0, abs(w)), (i, g, w)


@pytest.mark.parametrize("dt", [BF, F32])
def test_cp_decode_matches_the_oracle(mp, dt):
    # bf16: the tensor-core encoder's argmax epilogue; fp32: the CUDA-core encoder
    wl = small_workload(B=1, Hq=4, Hkv=2, n=2000, K=1, L=L_CP, kv_dtype=dt, q_dtype=dt,
                        w_dtype=dt)
    x = make_layer(wl)
    xc = {k: v.cuda() for k, v in x.items()}
    G = _rotations(L_CP, wl.d, 77, dt)
    Gc = G.cuda()
    table = mp.cp_logu_table(1, L_CP)
    centre = mp.key_mean(xc["keys"])
    codes = mp.encode_keys_cp(xc["keys"], centre, Gc, L_CP, 0, wl.n)
    args = (1, L_CP, wl.n_sink, wl.n_local)
    dbg = mp.debug_select(xc["q"], codes, centre, Gc, xc["keys"], xc["values"], *args,
                          counts=False, logu_table=table)
    prod = mp.decode_attention(xc["q"], codes, centre, Gc, xc["keys"], xc["values"], *args,
                               logu_table=table)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    assert torch.equal(prod, dbg["out"])
    gk = _unpack(codes, wl.B, wl.Hkv, wl.n, L_CP)
    qbytes = dbg["q_bits"].cpu().numpy().view(np.uint8).reshape(wl.B, wl.Hq, -1)[:, :, :L_CP]
    cen = centre.cpu().double().numpy()
    Gd = G.double().numpy()
    flips = rows = 0
    sizes = []
    for g in range(wl.Hkv):
        keys = O.as64(x["keys"][0, g])
        oc, alt, near = O.encode_keys_cp(keys, cen[0, g], Gd)
        kc, f = O.replay_codes(oc, alt, near, gk[0, g], what=f"key codes {g}")
        flips += f
        for h in range(g * wl.G, (g + 1) * wl.G):
            qv = O.as64(x["q"][0, h])
            qo, qa, qn = O.encode_query_cp(qv, Gd)
            qc, f = O.replay_codes(qo, qa, qn, qbytes[0, h][None, :].astype(np.int64),
                                   what=f"query codes {h}")
            flips += f
            r = O.decode_head(qv, keys, O.as64(x["values"][0, g]), cen[0, g], kc, qc[0], 1,
                              L_CP, wl.n_sink, wl.n_local, cross_polytope=True)
            cnt = int(dbg["sel_count"][0, h])
            got_S = dbg["sel_idx"][0, h, :cnt].cpu().numpy()
            assert np.array_equal(got_S, r["S"]), (h, cnt, r["S"].size)
            err = row_rel_err(dbg["out"][0, h].cpu().numpy(), r["o"])
            assert err <= OUT_REL_TOL, (h, err)
            rows += 1
            sizes.append(r["S"].size)
    assert rows == wl.Hq and flips <= 1e-4 * wl.Hkv * wl.n * L_CP
    assert 0.002 * wl.n < np.mean(sizes) < 0.2 * wl.n        # a few percent of the keys


def test_cp_ranges_and_spare_capacity(mp):
    # appends (ranges) give the codes of one pass; a cache with spare capacity decodes like the
    # contiguous one, bit for bit
    wl = small_workload(B=2, Hq=8, Hkv=2, n=2500, K=1, L=L_CP)
    xc = {k: v.cuda() for k, v in make_layer(wl).items()}
    G = _rotations(L_CP, wl.d, 78, BF).cuda()
    table = mp.cp_logu_table(1, L_CP)
    centre = mp.key_mean(xc["keys"])
    full = mp.encode_keys_cp(xc["keys"], centre, G, L_CP, 0, wl.n)
    parts = torch.zeros_like(full)
    for a, b in [(0, 700), (700, 701), (701, 1100), (1100, 2500)]:
        mp.encode_keys_cp(xc["keys"], centre, G, L_CP, a, b, parts)
    # the keys' bytes (the padding of the last block is not written)
    assert np.array_equal(_unpack(full, wl.B, wl.Hkv, wl.n, L_CP),
                          _unpack(parts, wl.B, wl.Hkv, wl.n, L_CP))
    args = (1, L_CP, wl.n_sink, wl.n_local)
    want = mp.decode_attention(xc["q"], full, centre, G, xc["keys"], xc["values"], *args,
                               logu_table=table)
    cap = 3500
    kc = torch.full((wl.B, wl.Hkv, cap, wl.d), 50.0, dtype=BF, device="cuda")
    vc = torch.full_like(kc, 50.0)
    kc[:, :, :wl.n] = xc["keys"]
    vc[:, :, :wl.n] = xc["values"]
    codes_c = mp.encode_keys_cp(kc, centre, G, L_CP, 0, wl.n)
    got = mp.decode_attention(xc["q"], codes_c, centre, G, kc, vc, *args, logu_table=table,
                              n=wl.n)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert mp.device_status() == 0


@pytest.mark.parametrize("shape", [
    dict(B=1, Hq=8, Hkv=1, n=1500, L=15),      # odd L: the last encoder chunk holds one table
    dict(B=2, Hq=2, Hkv=2, n=1100, L=3),       # no GQA, few tables, a ragged block
])
def test_cp_odd_tables_and_group_sizes(mp, shape):
    L = shape.pop("L")
    wl = small_workload(K=1, L=L, **shape)
    x = make_layer(wl)
    xc = {k: v.cuda() for k, v in x.items()}
    G = _rotations(L, wl.d, 79, BF)
    Gc = G.cuda()
    table = mp.cp_logu_table(1, L)
    centre = mp.key_mean(xc["keys"])
    codes = mp.encode_keys_cp(xc["keys"], centre, Gc, L, 0, wl.n)        # tensor cores
    simt = torch.zeros_like(codes)
    for a in range(0, wl.n, 64):                                          # CUDA cores
        mp.encode_keys_cp(xc["keys"], centre, Gc, L, a, min(wl.n, a + 64), simt)
    dbg = mp.debug_select(xc["q"], codes, centre, Gc, xc["keys"], xc["values"], 1, L,
                          wl.n_sink, wl.n_local, counts=False, logu_table=table)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    gk = _unpack(codes, wl.B, wl.Hkv, wl.n, L)
    gs = _unpack(simt, wl.B, wl.Hkv, wl.n, L)
    cen = centre.cpu().double().numpy()
    Gd = G.double().numpy()
    qbytes = dbg["q_bits"].cpu().numpy().view(np.uint8).reshape(wl.B, wl.Hq, -1)[:, :, :L]
    for b in range(wl.B):
        for g in range(wl.Hkv):
            keys = O.as64(x["keys"][b, g])
            oc, alt, near = O.encode_keys_cp(keys, cen[b, g], Gd)
            kc, _ = O.replay_codes(oc, alt, near, gk[b, g], what="tensor-core codes")
            O.replay_codes(oc, alt, near, gs[b, g], what="CUDA-core codes")
            for h in range(g * wl.G, (g + 1) * wl.G):
                qv = O.as64(x["q"][b, h])
                qo, qa, qn = O.encode_query_cp(qv, Gd)
                qc, _ = O.replay_codes(qo, qa, qn, qbytes[b, h][None, :].astype(np.int64))
                r = O.decode_head(qv, keys, O.as64(x["values"][b, g]), cen[b, g], kc, qc[0], 1, L,
                                  wl.n_sink, wl.n_local, cross_polytope=True)
                cnt = int(dbg["sel_count"][b, h])
                assert np.array_equal(dbg["sel_idx"][b, h, :cnt].cpu().numpy(), r["S"])
                assert row_rel_err(dbg["out"][b, h].cpu().numpy(), r["o"]) <= OUT_REL_TOL


def test_cp_full_96k_layer_against_the_oracle(mp):
    # the 96K workload's layer shape (B=1, 32 query heads over 8 KV heads, n = 98,304) with
    # L = 16 cross-polytope tables, encoded on the tensor cores; two KV heads checked
    wl = WORKLOADS["llama8b_n96k_32layers"].replace(K=1, L=L_CP)
    x = make_layer(wl, 0)
    xc = {k: v.cuda() for k, v in x.items()}
    G = _rotations(L_CP, wl.d, 78, BF)
    Gc = G.cuda()
    table = mp.cp_logu_table(1, L_CP)
    centre = mp.key_mean(xc["keys"])
    codes = mp.encode_keys_cp(xc["keys"], centre, Gc, L_CP, 0, wl.n)
    args = (1, L_CP, wl.n_sink, wl.n_local)
    dbg = mp.debug_select(xc["q"], codes, centre, Gc, xc["keys"], xc["values"], *args,
                          counts=False, logu_table=table)
    torch.cuda.synchronize()
    assert mp.device_status() == 0
    gk = _unpack(codes, wl.B, wl.Hkv, wl.n, L_CP)
    qbytes = dbg["q_bits"].cpu().numpy().view(np.uint8).reshape(wl.B, wl.Hq, -1)[:, :, :L_CP]
    cen = centre.cpu().double().numpy()
    Gd = G.double().numpy()
    flips = rows = 0
    for g in (0, 3):
        keys = O.as64(x["keys"][0, g])
        oc, alt, near = O.encode_keys_cp(keys, cen[0, g], Gd)
        kc, f = O.replay_codes(oc, alt, near, gk[0, g], what=f"key codes {g}")
        flips += f
        for h in range(g * wl.G, (g + 1) * wl.G):
            qv = O.as64(x["q"][0, h])
            qo, qa, qn = O.encode_query_cp(qv, Gd)
            qc, f = O.replay_codes(qo, qa, qn, qbytes[0, h][None, :].astype(np.int64),
                                   what=f"query codes {h}")
            flips += f
            r = O.decode_head(qv, keys, O.as64(x["values"][0, g]), cen[0, g], kc, qc[0], 1,
                              L_CP, wl.n_sink, wl.n_local, cross_polytope=True)
            cnt = int(dbg["sel_count"][0, h])
            assert np.array_equal(dbg["sel_idx"][0, h, :cnt].cpu().numpy(), r["S"]), (h, cnt)
            assert row_rel_err(dbg["out"][0, h].cpu().numpy(), r["o"]) <= OUT_REL_TOL, h
            rows += 1
    assert rows == 2 * wl.G and flips <= 1e-4 * 2 * wl.n * L_CP
