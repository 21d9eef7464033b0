"""GPU-vs-oracle parity checks (test infrastructure; imports the oracle).

What is compared, for one (sequence, KV head) unit and each query head of its GQA group:
  * key sign bits: GPU bits equal the oracle's everywhere outside the near-tie band
    |w_j.(k_i - mu)| < 1e-5 |w_j| |k_i|; inside it the GPU bit is replayed into the oracle
  * query sign bits: same rule with |w_j.q| < 1e-5 |w_j| |q|
  * collision counts (saturating at 255) and the sample set S: exact, after replay
  * the output row: max_e |o_gpu - o_ref| / max_e |o_ref| <= 1e-3 (fp32 accumulation on the GPU)
The bucketed decode is compared the same way, with the oracle's counts taken through its own
bucket tables (check_unit_buckets).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle as O

OUT_REL_TOL = 1e-3


def unpacked_to_bits(table_codes: np.ndarray, K: int) -> np.ndarray:
    """[n, L] per-table codes -> [n, K*L] bool, column t*K + b = bit b of table t."""
    tc = np.asarray(table_codes, dtype=np.int64)
    n, L = tc.shape
    if K == 0:
        return np.zeros((n, 0), dtype=bool)
    bits = (tc[:, :, None] >> np.arange(K)[None, None, :]) & 1
    return bits.reshape(n, L * K).astype(bool)


def words_to_bits(words: np.ndarray, C: int) -> np.ndarray:
    """[qwords] int32 words -> [C] bool, bit j%32 of word j/32."""
    w = np.asarray(words, dtype=np.int64) & 0xFFFFFFFF
    if C == 0:
        return np.zeros(0, dtype=bool)
    bits = (w[:, None] >> np.arange(32)[None, :]) & 1
    return bits.reshape(-1)[:C].astype(bool)


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.max(np.abs(ref)))
    num = float(np.max(np.abs(np.asarray(got, dtype=np.float64) - ref)))
    if den == 0.0:
        return num
    return num / den


@dataclasses.dataclass
class UnitReport:
    key_flips: int = 0
    q_flips: int = 0
    rows: int = 0
    max_rel_err: float = 0.0
    set_sizes: list = dataclasses.field(default_factory=list)


def check_unit(b: int, g: int, *, q, keys, values, centre, W, K, L, n_sink, n_local, gpu: dict,
               unpacked=None, scale=None, check_counts=True, radius=None) -> UnitReport:
    """Compare one (b, g) unit. q/keys/values/centre/W are the inputs both sides were given
    (torch tensors on any device, or arrays); gpu holds debug_select's outputs moved to the CPU
    and, when K > 0, the unpacked key codes [B, Hkv, n, L]. radius (the unit's longest centred
    key, as the GPU used it) selects the MIPS variant: W then has d + 1 rows."""
    rep = UnitReport()
    kb = O.as64(keys[b, g])
    vb = O.as64(values[b, g])
    mu = O.as64(centre[b, g])
    Hq = q.shape[1]
    Hkv = keys.shape[1]
    G = Hq // Hkv
    C = K * L
    Wd = O.as64(W)[:kb.shape[1]]                 # the query's rows (all of W but the MIPS row)
    if radius is None:
        _, obits, onear = O.encode_keys(kb, mu, W, K, L)
    else:
        _, obits, onear = O.encode_keys_mips(kb, mu, W, float(radius), K, L)
    if C:
        gbits = unpacked_to_bits(unpacked[b, g], K)
        kbits, rep.key_flips = O.replay_bits(obits, onear, gbits, what=f"key bits ({b},{g})")
    else:
        kbits = obits
    kcodes = O.table_codes(kbits, K, L)
    for h in range(g * G, (g + 1) * G):
        qv = O.as64(q[b, h])
        _, qb, qnear = O.encode_query(qv, Wd, K, L)
        gq = words_to_bits(gpu["q_bits"][b, h], C)
        qbits, f = O.replay_bits(qb[0], qnear[0], gq, what=f"query bits ({b},{h})")
        rep.q_flips += f
        qcode = O.table_codes(qbits[None, :], K, L)[0]
        r = O.decode_head(qv, kb, vb, mu, kcodes, qcode, K, L, n_sink, n_local, scale,
                          radius=None if radius is None else float(radius))
        if check_counts and gpu.get("cnt") is not None:
            want_cnt = np.minimum(r["cnt"], 255)
            got_cnt = np.asarray(gpu["cnt"][b, h], dtype=np.int64)
            bad = np.nonzero(want_cnt != got_cnt)[0]
            assert bad.size == 0, f"counts differ at ({b},{h}) keys {bad[:8].tolist()}"
        cnt_gpu = int(gpu["sel_count"][b, h])
        got_S = np.asarray(gpu["sel_idx"][b, h][:cnt_gpu], dtype=np.int64)
        assert np.array_equal(got_S, r["S"]), (
            f"sample set differs at ({b},{h}): gpu {cnt_gpu} keys, oracle {r['S'].size}; "
            f"only gpu {np.setdiff1d(got_S, r['S'])[:8].tolist()}, "
            f"only oracle {np.setdiff1d(r['S'], got_S)[:8].tolist()}")
        err = row_rel_err(gpu["out"][b, h], r["o"])
        assert err <= OUT_REL_TOL, f"output ({b},{h}) max relative error {err:.3e}"
        rep.rows += 1
        rep.max_rel_err = max(rep.max_rel_err, err)
        rep.set_sizes.append(int(r["S"].size))
    return rep


def _replayed_key_codes(b, g, keys, centre, W, K, L, unpacked, radius, rep):
    kb = O.as64(keys[b, g])
    mu = O.as64(centre[b, g])
    if radius is None:
        _, obits, onear = O.encode_keys(kb, mu, W, K, L)
    else:
        _, obits, onear = O.encode_keys_mips(kb, mu, W, float(radius), K, L)
    if K * L:
        gbits = unpacked_to_bits(unpacked[b, g], K)
        kbits, rep.key_flips = O.replay_bits(obits, onear, gbits, what=f"key bits ({b},{g})")
    else:
        kbits = obits
    return O.table_codes(kbits, K, L)


def check_unit_buckets(b: int, g: int, *, q, keys, values, centre, W, K, L, n_sink, n_local,
                       gpu: dict, unpacked, n_indexed=None, radius=None) -> UnitReport:
    """Compare one (b, g) unit of the bucketed decode (debug_select_buckets' outputs moved to the
    CPU) with the oracle's bucket route: the oracle builds its own tables (bucket_tables) of the
    codes of keys [0, n_indexed) after near-tie replay and counts each query's hits from them
    (bucket_collision_counts); keys of the blocks from n_indexed / 1024 on, which the decode scans,
    are counted directly. Sample sets exactly, outputs within 1e-3."""
    rep = UnitReport()
    kb = O.as64(keys[b, g])
    vb = O.as64(values[b, g])
    mu = O.as64(centre[b, g])
    n, d = kb.shape
    Hq, Hkv = q.shape[1], keys.shape[1]
    G = Hq // Hkv
    C = K * L
    ni = n if not n_indexed else int(n_indexed)
    tail0 = (ni // 1024) * 1024 if ni < n else n
    kcodes = _replayed_key_codes(b, g, keys, centre, W, K, L, unpacked, radius, rep)
    offsets, members = O.bucket_tables(kcodes[:ni], K, L)
    T = O.exact_set_mask(n, n_sink, n_local)
    Wd = O.as64(W)[:d]
    for h in range(g * G, (g + 1) * G):
        qv = O.as64(q[b, h])
        _, qb, qnear = O.encode_query(qv, Wd, K, L)
        gq = words_to_bits(gpu["q_bits"][b, h], C)
        qbits, f = O.replay_bits(qb[0], qnear[0], gq, what=f"query bits ({b},{h})")
        rep.q_flips += f
        qcode = O.table_codes(qbits[None, :], K, L)[0]
        cnt_direct = O.collision_counts(kcodes, qcode)
        cnt_tables = O.bucket_collision_counts(offsets, members, qcode, ni)
        assert np.array_equal(cnt_tables, cnt_direct[:ni]), "bucket and direct counts differ"
        cnt = np.concatenate([cnt_tables[:tail0], cnt_direct[tail0:]])
        S = O.sampled_set(cnt, T)
        r = O.decode_head(qv, kb, vb, mu, kcodes, qcode, K, L, n_sink, n_local,
                          radius=None if radius is None else float(radius))
        assert np.array_equal(r["S"], S)
        cnt_gpu = int(gpu["sel_count"][b, h])
        got_S = np.asarray(gpu["sel_idx"][b, h][:cnt_gpu], dtype=np.int64)
        assert np.array_equal(got_S, S), (
            f"bucketed sample set differs at ({b},{h}): gpu {cnt_gpu} keys, oracle {S.size}; "
            f"only gpu {np.setdiff1d(got_S, S)[:8].tolist()}, "
            f"only oracle {np.setdiff1d(S, got_S)[:8].tolist()}")
        err = row_rel_err(gpu["out"][b, h], r["o"])
        assert err <= OUT_REL_TOL, f"bucketed output ({b},{h}) max relative error {err:.3e}"
        rep.rows += 1
        rep.max_rel_err = max(rep.max_rel_err, err)
        rep.set_sizes.append(int(S.size))
    return rep


def run_gpu(lib, x: dict, centre, W, K, L, n_sink, n_local, scale=0.0, counts=True):
    """Build tables and run the debug and product decodes on the GPU; CPU copies of the results."""
    keys, values, q = x["keys"], x["values"], x["q"]
    B, Hkv, n, _ = keys.shape
    codes = lib.build_tables(keys, centre, W, K, L)
    dbg = lib.debug_select(q, codes, centre, W, keys, values, K, L, n_sink, n_local, scale,
                           counts=counts)
    prod = lib.decode_attention(q, codes, centre, W, keys, values, K, L, n_sink, n_local, scale)
    unpacked = lib.codes_unpack(codes, B, Hkv, n, K, L) if K * L else None
    torch.cuda.synchronize()
    out = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in dbg.items()}
    out["prod_out"] = prod.cpu().numpy()
    out["unpacked"] = unpacked.cpu().numpy() if unpacked is not None else None
    return out
