"""The seeded input generators: shapes, the geometry the recipe states, and stream stability."""
import torch

from workloads import WORKLOADS, make_layer, small_workload


def test_spread_keys_have_the_stated_covariance_and_leave_the_other_draws_alone():
    wl = small_workload(B=2, Hq=8, Hkv=2, n=3000, key_spread=16.0, key_spread_sigma=0.3,
                        index=77)
    x = make_layer(wl)
    base = make_layer(wl.replace(key_spread=0.0, key_spread_sigma=0.0))
    assert torch.equal(x["values"], base["values"]) and torch.equal(x["q"], base["q"])
    assert torch.equal(x["keys"][:, :, 0], base["keys"][:, :, 0])      # the sink is kept
    k = x["keys"].float()
    q = x["q"].float().view(2, 2, 4, 128).mean(dim=2)
    for b in range(2):
        for g in range(2):
            kk = k[b, g, 1:] - k[b, g, 1:].mean(0)
            evals, evecs = torch.linalg.eigh(kk.T @ kk / kk.shape[0])
            # 1 + a with a = 16 exp(N(0, 0.3^2)): within 4 sigma of the log-normal factor
            assert 1 + 16 * 0.3 < evals[-1] < 1 + 16 * 3.3
            assert evals[-2] < 1.7                  # the rest of the cone stays isotropic
            v = evecs[:, -1]
            cos = abs(float(v @ q[b, g] / q[b, g].norm()))
            assert cos > 0.7                        # the spread follows the group's queries


def test_workloads_have_the_recipe_shapes():
    wl = WORKLOADS["llama8b_b32_n32k_spread"]
    assert (wl.B, wl.Hq, wl.Hkv, wl.n, wl.K, wl.L) == (32, 32, 8, 32768, 10, 150)
    small = small_workload(B=1, Hq=4, Hkv=2, n=100)
    x = make_layer(small)
    assert x["keys"].shape == (1, 2, 100, 128) and x["q"].shape == (1, 4, 128)
    assert x["keys"].dtype == torch.bfloat16
