"""Child process of tests/test_gpu_checks.py: run with MAGICPIG_CHECKS=1 so that the binding loads
libmagicpig_checks.so, the build whose kernels check the indices of their global accesses and
raise MP_ERR_BOUNDS (status 6) instead of making an out-of-range one. Prints "checks ok" and
exits 0 when every assertion holds.

1. The decode (code scan) and the bucketed decode on clean inputs: no check fails and the results
   match the oracle (the same comparisons as the parity tests).
2. A bucket table corrupted the way a stray write would: the offsets of one table pointing past
   its n keys, the members of another holding a key index >= n. The bucketed lookup clamps the
   ranges and drops those members (in every build), and this build reports them: MP_ERR_BOUNDS
   with a bucket site. No access leaves the table: the offsets read are those of the query's
   code (< 2^K) and the members read lie below the clamped range end (<= n).
3. The status word resets and the next clean call stays clean.
4. The MIPS and cross-polytope variants (their encoder instantiations on the tensor cores, their
   decodes) on clean inputs: no check fails.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import lsh_sampled_sparse_gb300 as mp  # noqa: E402
from tests.parity import check_unit, check_unit_buckets, run_gpu  # noqa: E402
from workloads import make_hyperplanes, make_layer, small_workload  # noqa: E402

SITE_BUCKET_RANGE, SITE_BUCKET_KEY = 7, 8
MP_ERR_BOUNDS = 6


def main() -> None:
    assert os.environ.get("MAGICPIG_CHECKS") == "1"
    assert mp.library_path().endswith("libmagicpig_checks.so")
    enabled, site = mp.check_report()
    assert enabled and site == 0, (enabled, site)
    assert mp.device_status() == 0

    wl = small_workload(name="checks", index=730, B=2, Hq=8, Hkv=2, n=5000, K=10, L=150)
    xc = make_layer(wl)
    x = {k: v.cuda() for k, v in xc.items()}
    W = make_hyperplanes(wl)
    Wd = W.cuda()
    centre = mp.key_mean(x["keys"])
    args = (wl.K, wl.L, wl.n_sink, wl.n_local)

    # 1. clean inputs: the scan path and the bucketed path, against the oracle
    gpu = run_gpu(mp, x, centre, Wd, *args)
    assert mp.check_report() == (True, 0)
    for b in range(wl.B):
        for g in range(wl.Hkv):
            check_unit(b, g, q=xc["q"], keys=xc["keys"], values=xc["values"], centre=centre.cpu(),
                       W=W, K=wl.K, L=wl.L, n_sink=wl.n_sink, n_local=wl.n_local, gpu=gpu,
                       unpacked=gpu["unpacked"])
    codes = mp.build_tables(x["keys"], centre, Wd, wl.K, wl.L)
    buckets = mp.build_buckets(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L)
    dbg = mp.debug_select_buckets(x["q"], buckets, codes, centre, Wd, x["keys"], x["values"],
                                  *args)
    torch.cuda.synchronize()
    assert mp.check_report() == (True, 0)
    assert mp.device_status() == 0
    gb = {k: v.cpu().numpy() for k, v in dbg.items()}
    up = mp.codes_unpack(codes, wl.B, wl.Hkv, wl.n, wl.K, wl.L).cpu().numpy()
    for b in range(wl.B):
        for g in range(wl.Hkv):
            check_unit_buckets(b, g, q=xc["q"], keys=xc["keys"], values=xc["values"],
                               centre=centre.cpu(), W=W, K=wl.K, L=wl.L, n_sink=wl.n_sink,
                               n_local=wl.n_local, gpu=gb, unpacked=up)

    # 2. a corrupted table of head (0, 0): table 0's offsets past n, table 1's members >= n
    nb = 1 << wl.K
    bad = buckets.clone()
    bad[0:nb + 1] = wl.n + 1000
    m1 = wl.L * (nb + 1) + wl.n
    bad[m1:m1 + wl.n] = wl.n + 7
    ws = torch.empty(mp.decode_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.n, wl.d, *args),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(wl.B, wl.Hq, wl.d, dtype=torch.float32, device="cuda")
    mp.encode_query(x["q"], centre, Wd, x["keys"].shape, *args, ws)
    mp.sampled_attention_buckets(x["q"], bad, centre, x["keys"], x["values"], *args, out, ws)
    torch.cuda.synchronize()
    enabled, site = mp.check_report()
    assert enabled and site in (SITE_BUCKET_RANGE, SITE_BUCKET_KEY), site
    assert mp.device_status() == MP_ERR_BOUNDS
    assert torch.isfinite(out).all()

    # 3. the word was reset; a clean call stays clean
    assert mp.check_report() == (True, 0)
    mp.encode_query(x["q"], centre, Wd, x["keys"].shape, *args, ws)
    mp.sampled_attention_buckets(x["q"], buckets, centre, x["keys"], x["values"], *args, out, ws)
    torch.cuda.synchronize()
    assert mp.check_report() == (True, 0)
    assert mp.device_status() == 0

    # 4. the variants' encoders and decodes on clean inputs
    W_aug = torch.cat([Wd, torch.randn(1, Wd.shape[1], device="cuda").to(Wd.dtype)], 0).contiguous()
    radius = mp.key_radius(x["keys"], centre)
    mcodes = mp.encode_keys_mips(x["keys"], centre, W_aug, radius, wl.K, wl.L, 0, wl.n)
    mp.decode_attention(x["q"], mcodes, centre, W_aug, x["keys"], x["values"], *args,
                        radius=radius)
    L_cp = 16
    G = torch.randn(L_cp, wl.d, wl.d, device="cuda").to(torch.bfloat16).contiguous()
    table = mp.cp_logu_table(1, L_cp)
    ccodes = mp.encode_keys_cp(x["keys"], centre, G, L_cp, 0, wl.n)
    mp.decode_attention(x["q"], ccodes, centre, G, x["keys"], x["values"], 1, L_cp, wl.n_sink,
                        wl.n_local, logu_table=table)
    torch.cuda.synchronize()
    assert mp.check_report() == (True, 0)
    assert mp.device_status() == 0
    print("checks ok", flush=True)


if __name__ == "__main__":
    main()
