"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Codes, collision counts and sample sets must match exactly (sign bits may differ only inside the
near-tie band, where the GPU bit is replayed into the oracle); outputs within 1e-3 max relative
error per row. Small workloads are compared in full; the full-size workloads run on the GPU in
full and are compared on sampled (sequence, KV head) units the oracle can afford.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests.parity import check_unit, row_rel_err, run_gpu
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


def oracle_centre(keys, units=None, base=None):
    """Centre input: the oracle's fp64 mean rounded to fp32 for the given units (all if None);
    other units keep `base` (a plain fp64 mean taken on the device, never checked)."""
    B, Hkv, _, d = keys.shape
    c = base.clone().cpu() if base is not None else torch.zeros(B, Hkv, d)
    for b, g in (units or [(b, g) for b in range(B) for g in range(Hkv)]):
        c[b, g] = torch.tensor(O.key_centre(keys[b, g].cpu()), dtype=torch.float32)
    return c.float()


def run_case(mp, wl, *, x=None, W=None, centre=None, units=None, counts=True, layer=0):
    x = x if x is not None else make_layer(wl, layer)
    W = W if W is not None else make_hyperplanes(wl)
    centre = centre if centre is not None else oracle_centre(x["keys"])
    dev = {k: v.cuda() for k, v in x.items()}
    gpu = run_gpu(mp, dev, centre.cuda(), W.cuda(), wl.K, wl.L, wl.n_sink, wl.n_local,
                  counts=counts)
    assert np.array_equal(gpu["prod_out"], gpu["out"]), "debug and product decode differ"
    units = units or [(b, g) for b in range(wl.B) for g in range(wl.Hkv)]
    reps = [check_unit(b, g, q=x["q"], keys=x["keys"], values=x["values"], centre=centre,
                       W=W.cpu(), K=wl.K, L=wl.L, n_sink=wl.n_sink, n_local=wl.n_local, gpu=gpu,
                       unpacked=gpu["unpacked"], check_counts=counts) for b, g in units]
    return reps, gpu


def _summary(reps):
    return (sum(r.key_flips for r in reps), sum(r.q_flips for r in reps),
            max(r.max_rel_err for r in reps), sum(r.rows for r in reps))


# ------------------------------------------------------------------------------------------------
def test_key_mean_matches_oracle(mp):
    for dt, n in ((BF, 5000), (F32, 777), (BF, 98304)):
        wl = small_workload(B=2, Hq=3, Hkv=3, n=n, kv_dtype=dt)
        keys = make_layer(wl)["keys"]
        got = mp.key_mean(keys.cuda()).cpu().double().numpy()
        for b in range(2):
            for g in range(3):
                want = O.key_centre(keys[b, g])
                assert np.max(np.abs(got[b, g] - want)) <= 2e-6 * max(1.0, np.max(np.abs(want)))
    # run-to-run identical
    k = make_layer(small_workload(n=20000))["keys"].cuda()
    assert torch.equal(mp.key_mean(k), mp.key_mean(k))


def test_tiny_fp32_workload(mp):
    wl = WORKLOADS["tiny_f32_n4096"]
    reps, _ = run_case(mp, wl)
    kf, qf, err, rows = _summary(reps)
    assert rows == 1 and err <= 1e-3
    assert 0.01 < reps[0].set_sizes[0] / wl.n < 0.2       # centred cone: a few percent sampled


def test_llama8b_layer_b4_n16k(mp):
    wl = WORKLOADS["llama8b_b4_n16k"]
    reps, _ = run_case(mp, wl)
    kf, qf, err, rows = _summary(reps)
    assert rows == wl.B * wl.Hq
    total_bits = wl.B * wl.Hkv * wl.n * wl.C
    assert kf <= 1e-5 * total_bits, f"{kf} key near-tie flips"


@pytest.mark.parametrize("n,G,K,L,n_sink,n_local,dt,wdt", [
    (5000, 4, 10, 150, 4, 64, BF, BF),       # 4 full blocks + a ragged 904-key block
    (777, 2, 8, 75, 4, 64, BF, BF),          # one partial block
    (69, 1, 10, 150, 4, 64, BF, BF),         # one key outside T
    (2100, 8, 9, 120, 4, 64, BF, BF),        # GQA group of 8, (9, 120)
    (1100, 4, 11, 300, 4, 64, BF, BF),       # (11, 300): C = 3300 planes
    (3000, 4, 10, 150, 0, 0, BF, BF),        # empty exact set
    (4500, 1, 8, 75, 16, 200, F32, F32),     # fp32 everything, wide exact set
    (3000, 2, 10, 150, 4, 64, BF, F32),      # bf16 keys, fp32 hyperplanes (CUDA-core encoder)
    (1500, 2, 3, 5, 2, 3, BF, BF),           # tiny K, L: large sample sets
    (2048, 4, 10, 150, 1000, 1000, BF, BF),  # T spans several blocks
    (1024 * 9, 2, 10, 150, 4, 64, BF, BF),   # exact multiple of the block size
])
def test_shapes_and_edges(mp, n, G, K, L, n_sink, n_local, dt, wdt):
    wl = small_workload(B=2, Hq=2 * G, Hkv=2, n=n, K=K, L=L, n_sink=n_sink, n_local=n_local,
                        kv_dtype=dt, q_dtype=dt, w_dtype=wdt, index=200 + n % 97)
    reps, _ = run_case(mp, wl)
    assert _summary(reps)[2] <= 1e-3


def test_K0_selects_everything_and_is_full_attention(mp):
    wl = small_workload(B=1, Hq=4, Hkv=2, n=3000, K=0, L=4, index=301)
    x = make_layer(wl)
    reps, gpu = run_case(mp, wl, x=x)
    for h in range(wl.Hq):
        assert gpu["sel_count"][0, h] == wl.n - wl.n_sink - wl.n_local
        g = h // wl.G
        want = O.full_attention(x["q"][0, h], x["keys"][0, g], x["values"][0, g],
                                1 / np.sqrt(wl.d))
        assert row_rel_err(gpu["out"][0, h], want) <= 1e-3


def test_single_table_leaves_exact_set_only(mp):
    wl = small_workload(B=1, Hq=2, Hkv=1, n=4000, K=10, L=1, index=302)
    x = make_layer(wl)
    reps, gpu = run_case(mp, wl, x=x)
    T = np.nonzero(O.exact_set_mask(wl.n, wl.n_sink, wl.n_local))[0]
    for h in range(wl.Hq):
        assert gpu["sel_count"][0, h] == 0
        want = O.full_attention(x["q"][0, h], x["keys"][0, 0][T], x["values"][0, 0][T],
                                1 / np.sqrt(wl.d))
        assert row_rel_err(gpu["out"][0, h], want) <= 1e-3


@pytest.mark.parametrize("dt", [BF, F32])
def test_zero_query_and_key_at_centre(mp, dt):
    # zero-length q: every projection is 0, every bit 0 (strict >), cosine 0, p = 1/2;
    # a key exactly at the centre: k - mu = 0, cosine 0, p = 1/2
    wl = small_workload(B=1, Hq=2, Hkv=1, n=2500, index=303, kv_dtype=dt, q_dtype=dt,
                        w_dtype=dt)
    x = make_layer(wl)
    x["q"][0, 0] = 0.0
    centre = oracle_centre(x["keys"])
    centre = centre.to(torch.bfloat16).float()           # representable in either key dtype
    x["keys"][0, 0, 1000] = centre[0, 0].to(dt)
    reps, gpu = run_case(mp, wl, x=x, centre=centre)
    assert not np.any(gpu["q_bits"][0, 0])
    if dt == F32:                                        # fp32 path: k - mu is exactly 0
        assert not np.any(gpu["unpacked"][0, 0, 1000])


def test_outputs_are_deterministic(mp):
    wl = WORKLOADS["llama8b_b4_n16k"].replace(B=1)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    c = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], c, W, wl.K, wl.L)
    codes2 = mp.build_tables(x["keys"], c, W, wl.K, wl.L)
    assert torch.equal(codes, codes2)
    a = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], wl.K, wl.L, 4, 64)
    b = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], wl.K, wl.L, 4, 64)
    assert torch.equal(a, b)


def test_split_halves_equal_the_whole_decode(mp):
    wl = small_workload(B=2, Hq=8, Hkv=2, n=7000, index=305)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    c = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], c, W, wl.K, wl.L)
    ref = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], wl.K, wl.L, 4, 64)
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, wl.K, wl.L, 4,
                                               64), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(ref)
    mp.encode_query(x["q"], c, W, x["keys"].shape, wl.K, wl.L, 4, 64, ws)
    mp.sampled_attention(x["q"], codes, c, x["keys"], x["values"], wl.K, wl.L, 4, 64, out, ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_graph_capture_replays_the_same_step(mp):
    wl = small_workload(B=2, Hq=8, Hkv=2, n=6000, index=304)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    c = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], c, W, wl.K, wl.L)
    out = torch.empty(wl.B, wl.Hq, wl.d, device="cuda")
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, wl.K, wl.L, 4,
                                               64), dtype=torch.uint8, device="cuda")
    ref = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], wl.K, wl.L, 4, 64)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], wl.K, wl.L, 4, 64,
                                out=out, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ------------------------------------------------------------------------------------------------
# log u as the kernels evaluate it, against the oracle's fp64 binomial tail
# ------------------------------------------------------------------------------------------------
LOGU_ABS, LOGU_REL = 1e-4, 1e-6      # |log u_gpu - log u| <= 1e-4 + 1e-6 |log u|, c in (-1, 1]


@pytest.mark.parametrize("K,L", [(8, 75), (9, 120), (10, 150), (11, 300), (2, 3), (12, 2),
                                 (24, 2), (32, 5), (16, 10), (20, 1000)])
def test_log_inclusion_matches_the_oracle_over_the_cosine(mp, K, L):
    # the function every selected key's weight goes through ("LSH Sampling...", method details,
    # the u_i formula), as the attend kernel evaluates it (its per-call table, and the closed form
    # on the intervals where the table's chord is not close enough: few tables and many bits bend
    # log u sharply near cos = 1), at 10^4 grid cosines, 4,000 random ones and the range's ends
    rng = np.random.default_rng(400 + K)
    c = np.concatenate([-1.0 + 2.0 * np.arange(1, 10001) / 10000.0, rng.uniform(-1, 1, 4000),
                        1.0 - np.logspace(-7, -1, 200), -1.0 + np.logspace(-6, -1, 200)])
    c32 = torch.tensor(c, dtype=torch.float32)
    got = mp.debug_log_inclusion(c32.cuda(), K, L).cpu().double().numpy()
    cc = c32.double().numpy()                       # both sides at the same fp32 cosines
    p = 1.0 - np.arccos(cc) / np.pi
    want = O.log_inclusion_probability(p, K, L)
    err = np.abs(got - want)
    bound = LOGU_ABS + LOGU_REL * np.abs(want)
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), (f"c = {cc[worst]!r}: gpu {got[worst]!r}, oracle "
                                  f"{want[worst]!r}")
    # c = -1: p = 0, no collision is possible; the GPU clamps to log(FLT_MIN)
    at_m1 = mp.debug_log_inclusion(torch.tensor([-1.0], device="cuda"), K, L).item()
    assert at_m1 == pytest.approx(np.log(np.finfo(np.float32).tiny), rel=1e-6)


def test_log_inclusion_degenerate_parameters(mp):
    c = torch.linspace(-0.99, 1.0, 50, device="cuda")
    assert torch.all(mp.debug_log_inclusion(c, 0, 4) == 0.0)          # K = 0: u = 1
    assert torch.all(torch.isneginf(mp.debug_log_inclusion(c, 10, 1)))  # L = 1: u = 0


def test_nan_in_a_query_gives_a_nan_row_and_leaves_the_others(mp):
    wl = small_workload(B=2, Hq=8, Hkv=2, n=5000, index=306)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    c = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], c, W, wl.K, wl.L)
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)
    clean = mp.decode_attention(x["q"], codes, c, W, x["keys"], x["values"], *args)
    buckets = mp.build_buckets(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    q = x["q"].clone()
    q[1, 5, 17] = float("nan")
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, *args),
                     dtype=torch.uint8, device="cuda")
    scan = mp.decode_attention(q, codes, c, W, x["keys"], x["values"], *args)
    buck = torch.empty_like(scan)
    mp.encode_query(q, c, W, x["keys"].shape, *args, ws)
    mp.sampled_attention_buckets(q, buckets, c, x["keys"], x["values"], *args, buck, ws)
    torch.cuda.synchronize()
    assert mp.device_status() == 0                     # not a device-side failure
    keep = torch.ones(wl.B, wl.Hq, dtype=torch.bool)
    keep[1, 5] = False
    for out in (scan, buck):
        assert torch.all(torch.isnan(out[1, 5]))
        assert torch.all(torch.isfinite(out[keep.cuda()]))
    # the other rows keep their values; the NaN row's own selection changes the group's union
    # of rows, hence the order of some sums, so only up to rounding
    got, want = scan.cpu().numpy(), clean.cpu().numpy()
    for b in range(wl.B):
        for hh in range(wl.Hq):
            if keep[b, hh]:
                assert row_rel_err(got[b, hh], want[b, hh].astype(np.float64)) <= 1e-5


# ------------------------------------------------------------------------------------------------
# Full-size workloads: the whole layer runs on the GPU in the benchmark's launch configuration,
# the oracle checks sampled (sequence, KV head) units.
# ------------------------------------------------------------------------------------------------
def _full_size(mp, wl, units):
    x = make_layer(wl, 0, device="cuda")
    W = make_hyperplanes(wl, device="cuda")
    base = x["keys"].double().mean(dim=2).float()
    centre = oracle_centre(x["keys"], units=units, base=base)
    gpu_mean = mp.key_mean(x["keys"]).cpu()
    for b, g in units:
        want = centre[b, g].double()
        assert torch.max(torch.abs(gpu_mean[b, g].double() - want)) <= 2e-6 * max(1.0, float(
            want.abs().max()))
    reps, gpu = run_case(mp, wl, x=x, W=W, centre=centre, units=units)
    return reps


def test_full_size_llama8b_96k_layer(mp):
    wl = WORKLOADS["llama8b_n96k_32layers"]
    reps = _full_size(mp, wl, [(0, 0), (0, 5)])
    assert _summary(reps)[3] == 2 * wl.G


def test_full_size_b32_n32k(mp):
    wl = WORKLOADS["llama8b_b32_n32k"]
    reps = _full_size(mp, wl, [(0, 0), (17, 3), (31, 7)])
    assert _summary(reps)[3] == 3 * wl.G


def test_full_size_llama70b_layer(mp):
    wl = WORKLOADS["llama70b_b2_n128k_80layers"]
    reps = _full_size(mp, wl, [(1, 6)])
    assert _summary(reps)[3] == wl.G


def test_long_ragged_context_merges_75_partials(mp):
    """n = 300,000 (293 blocks, the last ragged): 74 sampled partials and the exact one per query
    head, so the last-arrival merge folds them in three passes of up to 32 (the 96K and 128K
    layers above take one and two)."""
    wl = small_workload(name="ctx300k", index=731, B=1, Hq=8, Hkv=2, n=300_000)
    reps = _full_size(mp, wl, [(0, 0), (0, 1)])
    assert _summary(reps)[3] == 2 * wl.G


def test_device_status_is_clean(mp):
    assert mp.device_status() == 0
