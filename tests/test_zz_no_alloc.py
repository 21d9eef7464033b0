"""mp_decode_attention_noalloc, the decode entry point that allocates nothing.

It serves callers that cannot allocate device memory when they call this library (a plugin
inside a runtime that owns all device memory through its own pool, a latency-critical loop
where an allocation may synchronise the device, code with no allocator at hand). Its scratch is
a fixed array inside the library, shared by every call. These tests call it through the C ABI
and check it against mp_decode_attention with a caller workspace, on consecutive calls of
different shapes (so a call must not depend on what the previous one left in the array): both
run the same kernels on the same inputs, so the outputs must be identical bit for bit. They also
cover the MIPS variant, and check that shapes too large for the array and the cross-polytope
variant are refused before anything runs.

The file is named so that pytest collects it after every other test file.
"""
import ctypes

import pytest
import torch

from workloads import make_hyperplanes, make_layer, small_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import lsh_sampled_sparse_gb300 as mp
    mp.lib()
    return mp


def _noalloc(mp, q, codes, centre, W, keys, values, wl, out, flags=0, radius=None, table=None):
    p = mp.Params(wl.K, wl.L, wl.n_sink, wl.n_local, 0.0, flags, 0, 0,
                  None if radius is None else radius.data_ptr(),
                  None if table is None else table.data_ptr())
    dt = {torch.bfloat16: mp.MP_BF16, torch.float32: mp.MP_F32}
    P = ctypes.c_void_p
    return mp.lib().mp_decode_attention_noalloc(
        P(q.data_ptr()), dt[q.dtype], P(codes.data_ptr()), P(centre.data_ptr()),
        P(W.data_ptr()), dt[W.dtype], P(keys.data_ptr()), P(values.data_ptr()), dt[keys.dtype],
        wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, ctypes.byref(p), P(out.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))


def _case(mp, wl):
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    W = make_hyperplanes(wl).cuda()
    centre = mp.key_mean(x["keys"])
    codes = mp.build_tables(x["keys"], centre, W, wl.K, wl.L)
    ref = mp.decode_attention(x["q"], codes, centre, W, x["keys"], x["values"], wl.K, wl.L,
                              wl.n_sink, wl.n_local)
    return x, W, centre, codes, ref


def test_noalloc_matches_the_workspace_decode_on_consecutive_calls(mp):
    first = small_workload(name="noalloc_a", index=950, B=1, Hq=32, Hkv=8, n=20000)
    second = small_workload(name="noalloc_b", index=951, B=2, Hq=8, Hkv=2, n=5000, K=8, L=75)
    cases = [(wl, _case(mp, wl)) for wl in (first, second)]
    for wl, (x, W, centre, codes, ref) in cases + cases[:1]:   # A, B, then A again
        out = torch.full_like(ref, float("nan"))
        status = _noalloc(mp, x["q"], codes, centre, W, x["keys"], x["values"], wl, out)
        assert status == 0, mp.lib().mp_status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)                   # same kernels, same inputs
        assert torch.all(torch.isfinite(out))
    assert mp.device_status() == 0


def test_noalloc_mips_variant_matches_the_workspace_decode(mp):
    wl = small_workload(name="noalloc_mips", index=953, B=1, Hq=8, Hkv=2, n=6000)
    x = {k: v.cuda() for k, v in make_layer(wl).items()}
    g = torch.Generator().manual_seed(953)
    W = torch.randn(wl.d + 1, wl.C, generator=g).to(torch.bfloat16).cuda()
    centre = mp.key_mean(x["keys"])
    radius = mp.key_radius(x["keys"], centre)
    codes = mp.encode_keys_mips(x["keys"], centre, W, radius, wl.K, wl.L, 0, wl.n)
    ref = mp.decode_attention(x["q"], codes, centre, W, x["keys"], x["values"], wl.K, wl.L,
                              wl.n_sink, wl.n_local, radius=radius)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        status = _noalloc(mp, x["q"], codes, centre, W, x["keys"], x["values"], wl, out,
                          flags=mp.MP_FLAG_MIPS, radius=radius)
        assert status == 0, mp.lib().mp_status_string(status)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert mp.device_status() == 0


def test_noalloc_refuses_the_cross_polytope_variant(mp):
    wl = small_workload(name="noalloc_cp", index=954, B=1, Hq=4, Hkv=1, n=3000, K=1, L=16)
    dev = "cuda"
    q = torch.zeros(wl.B, wl.Hq, wl.d, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(wl.B, wl.Hkv, wl.n, wl.d, dtype=torch.bfloat16, device=dev)
    centre = torch.zeros(wl.B, wl.Hkv, wl.d, device=dev)
    G = torch.zeros(wl.L, wl.d, wl.d, dtype=torch.bfloat16, device=dev)
    codes = torch.zeros(mp.cp_codes_bytes(wl.B, wl.Hkv, wl.n, wl.L) // 4, dtype=torch.int32,
                        device=dev)
    table = torch.zeros(mp.MP_LOGU_TABLE_ENTRIES, device=dev)
    out = torch.full((wl.B, wl.Hq, wl.d), 3.0, device=dev)
    status = _noalloc(mp, q, codes, centre, G, kv, kv, wl, out, flags=mp.MP_FLAG_CROSS_POLYTOPE,
                      table=table)
    assert status == 2                                   # MP_ERR_UNSUPPORTED, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


def test_noalloc_refuses_shapes_beyond_its_scratch(mp):
    # B=32 sequences at 32K context need about 17 MB of scratch, more than the 8 MiB array
    wl = small_workload(name="noalloc_big", index=952, B=32, Hq=32, Hkv=8, n=32768)
    need = mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, wl.K, wl.L, wl.n_sink,
                                     wl.n_local)
    assert need > 8 << 20
    dev = "cuda"
    q = torch.zeros(wl.B, wl.Hq, wl.d, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(wl.B, wl.Hkv, 64, wl.d, dtype=torch.bfloat16, device=dev)  # never read
    centre = torch.zeros(wl.B, wl.Hkv, wl.d, device=dev)
    W = torch.zeros(wl.d, wl.C, dtype=torch.bfloat16, device=dev)
    codes = torch.zeros(16, dtype=torch.int32, device=dev)
    out = torch.full((wl.B, wl.Hq, wl.d), 7.0, device=dev)
    status = _noalloc(mp, q, codes, centre, W, kv, kv, wl, out)
    assert status == 5                                   # MP_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
