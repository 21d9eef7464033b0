"""ctypes binding of libmagicpig: argument checks and marshalling only.

Names follow the C ABI in include/magicpig.h without the ``mp_`` prefix. Tensors are PyTorch CUDA
tensors; outputs and workspaces are allocated here with PyTorch when the caller passes none.
Packed codes and bit vectors are held in int32 tensors (the same bits as the ABI's uint32).
"""
from __future__ import annotations

import ctypes
import os

import torch

MP_F32, MP_BF16 = 0, 1
_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p


class MagicPIGError(RuntimeError):
    """A libmagicpig call returned a status other than MP_OK, or the library is missing."""


MP_FLAG_MIPS = 1
MP_FLAG_CROSS_POLYTOPE = 2
MP_LOGU_TABLE_ENTRIES = 4097


class Params(ctypes.Structure):
    """mp_params: K bits per table, L tables, exact sink/local sizes, score scale (0: 1/sqrt(d)),
    flags (0, MP_FLAG_MIPS or MP_FLAG_CROSS_POLYTOPE), the cache capacity per head (0: n), the
    keys in the bucketed tables (0: n), the MIPS variant's radii and the cross-polytope variant's
    log u table (device pointers, or None)."""

    _fields_ = [("K", ctypes.c_int), ("L", ctypes.c_int), ("n_sink", ctypes.c_int),
                ("n_local", ctypes.c_int), ("scale", ctypes.c_float), ("flags", ctypes.c_uint),
                ("n_capacity", ctypes.c_int), ("n_indexed", ctypes.c_int),
                ("radius", ctypes.c_void_p), ("logu_table", ctypes.c_void_p)]


def _params(K, L, n_sink, n_local, scale=0.0, n_capacity=0, n_indexed=0, radius=None,
            logu_table=None) -> Params:
    flags = 0
    for t, name, flag in ((radius, "radius", MP_FLAG_MIPS),
                          (logu_table, "logu_table", MP_FLAG_CROSS_POLYTOPE)):
        if t is not None:
            _cuda(t, name)
            if t.dtype != torch.float32:
                raise TypeError(f"{name} must be float32")
            flags |= flag
    return Params(K, L, n_sink, n_local, scale, flags, n_capacity, n_indexed,
                  None if radius is None else radius.data_ptr(),
                  None if logu_table is None else logu_table.data_ptr())


def _lengths(keys_shape, n):
    """(n, n_capacity) of a cache tensor [B, Hkv, n_capacity, d] of which n keys are in use."""
    cap = int(keys_shape[2])
    if n is None:
        return cap, cap
    if not 1 <= n <= cap:
        raise ValueError(f"n = {n} outside [1, {cap}] (the cache's capacity)")
    return int(n), cap


_LIB = None


def library_path() -> str:
    """libmagicpig.so, or with MAGICPIG_CHECKS=1 in the environment the MP_CHECKS build
    libmagicpig_checks.so (python -m lsh_sampled_sparse_gb300.build --checks)."""
    name = "libmagicpig_checks.so" if os.environ.get("MAGICPIG_CHECKS") == "1" \
        else "libmagicpig.so"
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), name)


def _declare(L):
    P = ctypes.POINTER(Params)
    sig = {
        "mp_status_string": (ctypes.c_char_p, [_c_int]),
        "mp_abi_version": (_c_int, []),
        "mp_codes_bytes": (_c_size, [_c_int] * 5),
        "mp_key_mean_workspace_bytes": (_c_size, [_c_int] * 4),
        "mp_key_mean": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _c_size,
                                 _vp]),
        "mp_key_mean_cap": (_c_int, [_vp, _c_int] + [_c_int] * 5 + [_vp, _vp, _c_size, _vp]),
        "mp_encode_keys": (_c_int, [_vp, _c_int, _vp, _vp, _c_int] + [_c_int] * 8 + [_vp, _vp]),
        "mp_key_radius": (_c_int, [_vp, _c_int, _vp] + [_c_int] * 5 + [_vp, _vp]),
        "mp_cp_codes_bytes": (_c_size, [_c_int] * 4),
        "mp_cp_logu_table": (_c_int, [_c_int] * 3 + [_vp, _vp]),
        "mp_encode_keys_cp": (_c_int, [_vp, _c_int, _vp, _vp, _c_int] + [_c_int] * 7 + [_vp, _vp]),
        "mp_encode_keys_mips": (_c_int, [_vp, _c_int, _vp, _vp, _c_int, _vp] + [_c_int] * 8
                                + [_vp, _vp, _vp]),
        "mp_build_tables": (_c_int, [_vp, _c_int, _vp, _vp, _c_int] + [_c_int] * 6 + [_vp, _vp]),
        "mp_decode_workspace_bytes": (_c_size, [_c_int] * 5 + [P]),
        "mp_debug_workspace_bytes": (_c_size, [_c_int] * 5 + [P]),
        "mp_decode_attention": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp, _c_int]
                                + [_c_int] * 5 + [P, _vp, _vp, _c_size, _vp]),
        "mp_encode_query": (_c_int, [_vp, _c_int, _vp, _vp, _c_int] + [_c_int] * 5
                            + [P, _vp, _c_size, _vp]),
        "mp_sampled_attention": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _c_int]
                                 + [_c_int] * 5 + [P, _vp, _vp, _c_size, _vp]),
        "mp_debug_select": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp, _c_int]
                            + [_c_int] * 5 + [P, _vp, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
        "mp_decode_attention_noalloc": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _c_int, _vp, _vp,
                                                 _c_int] + [_c_int] * 5 + [P, _vp, _vp]),
        "mp_codes_unpack": (_c_int, [_vp] + [_c_int] * 5 + [_vp, _vp]),
        "mp_buckets_bytes": (_c_size, [_c_int] * 5),
        "mp_build_buckets": (_c_int, [_vp] + [_c_int] * 5 + [_vp, _vp]),
        "mp_build_buckets_cap": (_c_int, [_vp] + [_c_int] * 6 + [_vp, _vp]),
        "mp_sampled_attention_buckets": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int]
                                         + [_c_int] * 5 + [P, _vp, _vp, _c_size, _vp]),
        "mp_debug_select_buckets": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _c_int, _vp, _vp,
                                             _c_int] + [_c_int] * 5
                                    + [P, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
        "mp_debug_log_inclusion": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _vp]),
        "mp_debug_wait_expiry": (_c_int, [_c_int, _vp]),
        "mp_device_status": (_c_int, [ctypes.POINTER(_c_int)]),
        "mp_debug_check_report": (_c_int, [ctypes.POINTER(_c_int), ctypes.POINTER(_c_int)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def lib():
    """The loaded libmagicpig (raises MagicPIGError if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise MagicPIGError(
                f"{path} is missing; build it with `python -m lsh_sampled_sparse_gb300.build`."
                " There is no CPU fallback.")
        handle = ctypes.CDLL(path)
        _declare(handle)
        _LIB = handle
    return _LIB


def abi_version() -> int:
    return int(lib().mp_abi_version())


def _check(status: int, what: str) -> None:
    if status != 0:
        raise MagicPIGError(f"{what} failed: {lib().mp_status_string(status).decode()}")


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream)


def _dtype(t: torch.Tensor, name: str) -> int:
    if t.dtype == torch.bfloat16:
        return MP_BF16
    if t.dtype == torch.float32:
        return MP_F32
    raise TypeError(f"{name}: dtype {t.dtype} is not float32 or bfloat16")


def _cuda(t, name: str, ndim: int | None = None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    return t


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _workspace(ws, nbytes: int, device):
    if ws is None:
        return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _cuda(ws, "workspace")
    if _nbytes(ws) < nbytes:
        raise ValueError(f"workspace has {_nbytes(ws)} bytes, needs {nbytes}")
    return ws


def codes_bytes(B: int, Hkv: int, n: int, K: int, L: int) -> int:
    return int(lib().mp_codes_bytes(B, Hkv, n, K, L))


def key_mean_workspace_bytes(B: int, Hkv: int, n: int, d: int) -> int:
    return int(lib().mp_key_mean_workspace_bytes(B, Hkv, n, d))


def decode_workspace_bytes(B, Hq, Hkv, n, d, K, L, n_sink, n_local, scale=0.0, radius=None,
                           logu_table=None) -> int:
    """Workspace bytes of a decode with these shapes (and variant: pass the variant's radius or
    log u table as the decode will)."""
    p = _params(K, L, n_sink, n_local, scale, radius=radius, logu_table=logu_table)
    return int(lib().mp_decode_workspace_bytes(B, Hq, Hkv, n, d, ctypes.byref(p)))


def debug_workspace_bytes(B, Hq, Hkv, n, d, K, L, n_sink, n_local, scale=0.0) -> int:
    p = _params(K, L, n_sink, n_local, scale)
    return int(lib().mp_debug_workspace_bytes(B, Hq, Hkv, n, d, ctypes.byref(p)))


def key_mean(keys, centre=None, workspace=None, stream=None, n=None):
    """mu[b, g] = mean of the first n keys of keys[b, g] (float32 [B, Hkv, d]); n defaults to
    keys.shape[2], a larger keys.shape[2] is the cache's capacity."""
    _cuda(keys, "keys", 4)
    B, Hkv, cap, d = keys.shape
    n, cap = _lengths(keys.shape, n)
    if centre is None:
        centre = torch.empty(B, Hkv, d, dtype=torch.float32, device=keys.device)
    _cuda(centre, "centre", 3)
    ws = _workspace(workspace, key_mean_workspace_bytes(B, Hkv, n, d), keys.device)
    _check(lib().mp_key_mean_cap(_ptr(keys), _dtype(keys, "keys"), B, Hkv, cap, n, d,
                                 _ptr(centre), _ptr(ws), _nbytes(ws), _stream(stream)),
           "mp_key_mean_cap")
    return centre


def build_tables(keys, centre, W, K: int, L: int, codes=None, stream=None):
    """Packed bit-sliced SimHash codes of every key (int32 tensor of codes_bytes/4 words)."""
    _cuda(keys, "keys", 4)
    B, Hkv, n, d = keys.shape
    nbytes = codes_bytes(B, Hkv, n, K, L)
    if codes is None:
        codes = torch.empty(max(nbytes // 4, 4), dtype=torch.int32, device=keys.device)
    _cuda(codes, "codes")
    if _nbytes(codes) < nbytes:
        raise ValueError("codes buffer too small")
    _cuda(centre, "centre", 3)
    _cuda(W, "W", 2)
    _check(lib().mp_build_tables(_ptr(keys), _dtype(keys, "keys"), _ptr(centre), _ptr(W),
                                 _dtype(W, "W"), B, Hkv, n, d, K, L, _ptr(codes),
                                 _stream(stream)), "mp_build_tables")
    return codes


def encode_keys(keys, centre, W, K: int, L: int, n_begin: int, n_end: int, codes,
                stream=None):
    """(Re)encode keys [n_begin, n_end) of the cache keys [B, Hkv, n_capacity, d] into codes laid
    out for n_capacity (the incremental append of decode tokens)."""
    _cuda(keys, "keys", 4)
    B, Hkv, cap, d = keys.shape
    _cuda(codes, "codes")
    if _nbytes(codes) < codes_bytes(B, Hkv, cap, K, L):
        raise ValueError("codes buffer too small for the cache's capacity")
    _cuda(centre, "centre", 3)
    _cuda(W, "W", 2)
    _check(lib().mp_encode_keys(_ptr(keys), _dtype(keys, "keys"), _ptr(centre), _ptr(W),
                                _dtype(W, "W"), B, Hkv, cap, n_begin, n_end, d, K, L,
                                _ptr(codes), _stream(stream)), "mp_encode_keys")
    return codes


def key_radius(keys, centre, n=None, radius=None, stream=None):
    """MIPS variant: radius[b, g] = max over the first n keys of |k - mu| (float32 [B, Hkv])."""
    _cuda(keys, "keys", 4)
    _cuda(centre, "centre", 3)
    B, Hkv, cap, d = keys.shape
    n, cap = _lengths(keys.shape, n)
    if radius is None:
        radius = torch.empty(B, Hkv, dtype=torch.float32, device=keys.device)
    _cuda(radius, "radius")
    _check(lib().mp_key_radius(_ptr(keys), _dtype(keys, "keys"), _ptr(centre), B, Hkv, cap, n, d,
                               _ptr(radius), _stream(stream)), "mp_key_radius")
    return radius


def encode_keys_mips(keys, centre, W_aug, radius, K: int, L: int, n_begin: int, n_end: int,
                     codes=None, stream=None, tensor_cores: bool = True, norms_scratch=None):
    """MIPS variant: codes of keys [n_begin, n_end) from the keys extended by
    sqrt(r^2 - |k - mu|^2), W_aug [d + 1, K*L]; codes laid out for keys.shape[2] keys per head.
    tensor_cores: let long bf16 ranges run on the tensor-core encoder (a scratch of one float
    per cached key is allocated unless norms_scratch is given)."""
    _cuda(keys, "keys", 4)
    B, Hkv, cap, d = keys.shape
    nbytes = codes_bytes(B, Hkv, cap, K, L)
    if codes is None:
        codes = torch.empty(max(nbytes // 4, 4), dtype=torch.int32, device=keys.device)
    _cuda(codes, "codes")
    if _nbytes(codes) < nbytes:
        raise ValueError("codes buffer too small for the cache's capacity")
    _cuda(centre, "centre", 3)
    _cuda(W_aug, "W_aug", 2)
    _cuda(radius, "radius")
    if W_aug.shape[0] != d + 1:
        raise ValueError("W_aug must have d + 1 rows")
    scratch = None
    if tensor_cores:
        scratch = norms_scratch
        if scratch is None:
            scratch = torch.empty(B * Hkv * cap, dtype=torch.float32, device=keys.device)
        _cuda(scratch, "norms_scratch")
        if _nbytes(scratch) < B * Hkv * cap * 4:
            raise ValueError("norms_scratch needs one float per cached key")
    _check(lib().mp_encode_keys_mips(_ptr(keys), _dtype(keys, "keys"), _ptr(centre), _ptr(W_aug),
                                     _dtype(W_aug, "W_aug"), _ptr(radius), B, Hkv, cap, n_begin,
                                     n_end, d, K, L, _ptr(codes), _ptr(scratch),
                                     _stream(stream)), "mp_encode_keys_mips")
    return codes


def cp_codes_bytes(B: int, Hkv: int, n: int, L: int) -> int:
    return int(lib().mp_cp_codes_bytes(B, Hkv, n, L))


def cp_logu_table(K: int, L: int, table=None, d: int = 128, stream=None):
    """Cross-polytope variant: log u at MP_LOGU_TABLE_ENTRIES cosines on [-1, 1] (float32)."""
    if table is None:
        table = torch.empty(MP_LOGU_TABLE_ENTRIES, dtype=torch.float32, device="cuda")
    _cuda(table, "table")
    if table.numel() < MP_LOGU_TABLE_ENTRIES or table.dtype != torch.float32:
        raise ValueError("the table needs MP_LOGU_TABLE_ENTRIES float32 entries")
    _check(lib().mp_cp_logu_table(K, L, d, _ptr(table), _stream(stream)), "mp_cp_logu_table")
    return table


def encode_keys_cp(keys, centre, G, L: int, n_begin: int, n_end: int, codes=None, stream=None):
    """Cross-polytope variant: byte codes of keys [n_begin, n_end) (G [L, d, d]); codes laid out
    for keys.shape[2] keys per head."""
    _cuda(keys, "keys", 4)
    B, Hkv, cap, d = keys.shape
    nbytes = cp_codes_bytes(B, Hkv, cap, L)
    if codes is None:
        codes = torch.empty(nbytes, dtype=torch.uint8, device=keys.device)
    _cuda(codes, "codes")
    if _nbytes(codes) < nbytes:
        raise ValueError("codes buffer too small for the cache's capacity")
    _cuda(centre, "centre", 3)
    _cuda(G, "G", 3)
    _check(lib().mp_encode_keys_cp(_ptr(keys), _dtype(keys, "keys"), _ptr(centre), _ptr(G),
                                   _dtype(G, "G"), B, Hkv, cap, n_begin, n_end, d, L,
                                   _ptr(codes), _stream(stream)), "mp_encode_keys_cp")
    return codes


def decode_attention(q, codes, centre, W, keys, values, K: int, L: int, n_sink: int,
                     n_local: int, scale: float = 0.0, out=None, workspace=None, stream=None,
                     n=None, radius=None, logu_table=None):
    """One LSH-sampled decode step over the first n keys (default: all of keys.shape[2]);
    returns out [B, Hq, d] float32."""
    _cuda(q, "q", 3)
    _cuda(keys, "keys", 4)
    _cuda(values, "values", 4)
    _cuda(centre, "centre", 3)
    B, Hq, d = q.shape
    Hkv = keys.shape[1]
    n, cap = _lengths(keys.shape, n)
    if values.shape != keys.shape or values.dtype != keys.dtype:
        raise ValueError("values must match keys in shape and dtype")
    if out is None:
        out = torch.empty(B, Hq, d, dtype=torch.float32, device=q.device)
    _cuda(out, "out", 3)
    p = _params(K, L, n_sink, n_local, scale, cap, radius=radius, logu_table=logu_table)
    need = int(lib().mp_decode_workspace_bytes(B, Hq, Hkv, n, d, ctypes.byref(p)))
    if need == 0:
        raise MagicPIGError("mp_decode_workspace_bytes rejected the shapes/parameters")
    ws = _workspace(workspace, need, q.device)
    _check(lib().mp_decode_attention(
        _ptr(q), _dtype(q, "q"), _ptr(codes), _ptr(centre), _ptr(W), _dtype(W, "W"), _ptr(keys),
        _ptr(values), _dtype(keys, "keys"), B, Hq, Hkv, n, d, ctypes.byref(p), _ptr(out),
        _ptr(ws), _nbytes(ws), _stream(stream)), "mp_decode_attention")
    return out


def encode_query(q, centre, W, keys_shape, K: int, L: int, n_sink: int, n_local: int,
                 workspace, scale: float = 0.0, stream=None, n=None, radius=None,
                 logu_table=None):
    """First half of decode_attention: query codes and norms into `workspace`."""
    _cuda(q, "q", 3)
    _cuda(centre, "centre", 3)
    _cuda(workspace, "workspace")
    B, Hq, d = q.shape
    Hkv = keys_shape[1]
    n, cap = _lengths(keys_shape, n)
    p = _params(K, L, n_sink, n_local, scale, cap, radius=radius, logu_table=logu_table)
    _check(lib().mp_encode_query(_ptr(q), _dtype(q, "q"), _ptr(centre), _ptr(W), _dtype(W, "W"),
                                 B, Hq, Hkv, n, d, ctypes.byref(p), _ptr(workspace),
                                 _nbytes(workspace), _stream(stream)), "mp_encode_query")


def sampled_attention(q, codes, centre, keys, values, K: int, L: int, n_sink: int, n_local: int,
                      out, workspace, scale: float = 0.0, stream=None, n=None, radius=None,
                      logu_table=None):
    """Second half of decode_attention (after encode_query filled `workspace`)."""
    _cuda(q, "q", 3)
    _cuda(keys, "keys", 4)
    _cuda(values, "values", 4)
    _cuda(out, "out", 3)
    _cuda(workspace, "workspace")
    B, Hq, d = q.shape
    Hkv = keys.shape[1]
    n, cap = _lengths(keys.shape, n)
    p = _params(K, L, n_sink, n_local, scale, cap, radius=radius, logu_table=logu_table)
    _check(lib().mp_sampled_attention(
        _ptr(q), _dtype(q, "q"), _ptr(codes), _ptr(centre), _ptr(keys), _ptr(values),
        _dtype(keys, "keys"), B, Hq, Hkv, n, d, ctypes.byref(p), _ptr(out), _ptr(workspace),
        _nbytes(workspace), _stream(stream)), "mp_sampled_attention")
    return out


def buckets_bytes(B: int, Hkv: int, n: int, K: int, L: int) -> int:
    return int(lib().mp_buckets_bytes(B, Hkv, n, K, L))


def build_buckets(codes, B: int, Hkv: int, n: int, K: int, L: int, buckets=None, stream=None,
                  n_capacity=None):
    """Bucketed hash tables of keys [0, n) from the packed codes (laid out for n_capacity keys
    per head, default n); an int32 tensor of buckets_bytes/4 words."""
    nbytes = buckets_bytes(B, Hkv, n, K, L)
    if nbytes == 0:
        raise ValueError("unsupported bucket table shape (K must be <= 12)")
    if buckets is None:
        buckets = torch.empty(nbytes // 4, dtype=torch.int32, device=codes.device)
    _cuda(codes, "codes")
    _cuda(buckets, "buckets")
    if _nbytes(buckets) < nbytes:
        raise ValueError("buckets buffer too small")
    cap = n if n_capacity is None else int(n_capacity)
    _check(lib().mp_build_buckets_cap(_ptr(codes), B, Hkv, cap, n, K, L, _ptr(buckets),
                                      _stream(stream)), "mp_build_buckets_cap")
    return buckets


def sampled_attention_buckets(q, buckets, centre, keys, values, K: int, L: int, n_sink: int,
                              n_local: int, out, workspace, scale: float = 0.0, stream=None,
                              codes=None, n=None, n_indexed=None, radius=None):
    """sampled_attention with the bucketed tables in place of the code scan. The tables hold
    keys [0, n_indexed) (default n); keys appended since are found by scanning their codes, so
    `codes` is needed when n_indexed < n."""
    _cuda(q, "q", 3)
    _cuda(keys, "keys", 4)
    _cuda(values, "values", 4)
    _cuda(out, "out", 3)
    _cuda(workspace, "workspace")
    _cuda(buckets, "buckets")
    B, Hq, d = q.shape
    Hkv = keys.shape[1]
    n, cap = _lengths(keys.shape, n)
    p = _params(K, L, n_sink, n_local, scale, cap, 0 if n_indexed is None else int(n_indexed),
                radius=radius)
    _check(lib().mp_sampled_attention_buckets(
        _ptr(q), _dtype(q, "q"), _ptr(buckets), _ptr(codes), _ptr(centre), _ptr(keys),
        _ptr(values), _dtype(keys, "keys"), B, Hq, Hkv, n, d, ctypes.byref(p), _ptr(out),
        _ptr(workspace), _nbytes(workspace), _stream(stream)), "mp_sampled_attention_buckets")
    return out


def debug_select(q, codes, centre, W, keys, values, K: int, L: int, n_sink: int, n_local: int,
                 scale: float = 0.0, counts: bool = True, stream=None, n=None,
                 radius=None, logu_table=None) -> dict:
    """Decode plus its decisions: out, q_bits, per-row ascending sample sets, collision counts."""
    _cuda(q, "q", 3)
    _cuda(keys, "keys", 4)
    B, Hq, d = q.shape
    Hkv = keys.shape[1]
    n, cap = _lengths(keys.shape, n)
    dev = q.device
    C = K * L
    qwords = (C + 31) // 32 if logu_table is None else (L + 3) // 4   # bits, or code bytes
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    q_bits = torch.zeros(B, Hq, max(qwords, 1), dtype=torch.int32, device=dev)
    sel_idx = torch.full((B, Hq, n), -1, dtype=torch.int32, device=dev)
    sel_count = torch.zeros(B, Hq, dtype=torch.int32, device=dev)
    cnt = torch.zeros(B, Hq, n, dtype=torch.uint8, device=dev) if counts else None
    p = _params(K, L, n_sink, n_local, scale, cap, radius=radius, logu_table=logu_table)
    need = int(lib().mp_debug_workspace_bytes(B, Hq, Hkv, n, d, ctypes.byref(p)))
    if need == 0:
        raise MagicPIGError("mp_debug_workspace_bytes rejected the shapes/parameters")
    ws = _workspace(None, need, dev)
    _check(lib().mp_debug_select(
        _ptr(q), _dtype(q, "q"), _ptr(codes), _ptr(centre), _ptr(W), _dtype(W, "W"), _ptr(keys),
        _ptr(values), _dtype(keys, "keys"), B, Hq, Hkv, n, d, ctypes.byref(p), _ptr(out),
        _ptr(q_bits) if qwords else None, _ptr(sel_idx), _ptr(sel_count), _ptr(cnt), _ptr(ws),
        _nbytes(ws), _stream(stream)), "mp_debug_select")
    return {"out": out, "q_bits": q_bits[..., :qwords], "sel_idx": sel_idx,
            "sel_count": sel_count, "cnt": cnt}


def debug_select_buckets(q, buckets, codes, centre, W, keys, values, K: int, L: int,
                         n_sink: int, n_local: int, scale: float = 0.0, stream=None, n=None,
                         n_indexed: int = 0, radius=None) -> dict:
    """The bucketed decode plus its decisions: out, q_bits, per-row ascending sample sets."""
    _cuda(q, "q", 3)
    _cuda(keys, "keys", 4)
    _cuda(buckets, "buckets")
    B, Hq, d = q.shape
    Hkv = keys.shape[1]
    n, cap = _lengths(keys.shape, n)
    dev = q.device
    qwords = (K * L + 31) // 32
    out = torch.empty(B, Hq, d, dtype=torch.float32, device=dev)
    q_bits = torch.zeros(B, Hq, max(qwords, 1), dtype=torch.int32, device=dev)
    sel_idx = torch.full((B, Hq, n), -1, dtype=torch.int32, device=dev)
    sel_count = torch.zeros(B, Hq, dtype=torch.int32, device=dev)
    p = _params(K, L, n_sink, n_local, scale, cap, n_indexed, radius=radius)
    need = int(lib().mp_debug_workspace_bytes(B, Hq, Hkv, n, d, ctypes.byref(p)))
    if need == 0:
        raise MagicPIGError("mp_debug_workspace_bytes rejected the shapes/parameters")
    ws = _workspace(None, need, dev)
    _check(lib().mp_debug_select_buckets(
        _ptr(q), _dtype(q, "q"), _ptr(buckets), _ptr(codes), _ptr(centre), _ptr(W),
        _dtype(W, "W"), _ptr(keys), _ptr(values), _dtype(keys, "keys"), B, Hq, Hkv, n, d,
        ctypes.byref(p), _ptr(out), _ptr(q_bits) if qwords else None, _ptr(sel_idx),
        _ptr(sel_count), _ptr(ws), _nbytes(ws), _stream(stream)), "mp_debug_select_buckets")
    return {"out": out, "q_bits": q_bits[..., :qwords], "sel_idx": sel_idx,
            "sel_count": sel_count}


def debug_log_inclusion(cosines, K: int, L: int, out=None, stream=None):
    """log u at each cosine (float32 CUDA tensor), as the decode kernels evaluate it."""
    _cuda(cosines, "cosines")
    if cosines.dtype != torch.float32:
        raise TypeError("cosines must be float32")
    out = torch.empty_like(cosines) if out is None else out
    _check(lib().mp_debug_log_inclusion(_ptr(cosines), cosines.numel(), K, L, _ptr(out),
                                        _stream(stream)), "mp_debug_log_inclusion")
    return out


def debug_wait_expiry(limit_us: int, stream=None) -> None:
    """Run the failure path's test hook: a bounded wait that gives up after limit_us."""
    _check(lib().mp_debug_wait_expiry(int(limit_us), _stream(stream)), "mp_debug_wait_expiry")


def codes_unpack(codes, B: int, Hkv: int, n: int, K: int, L: int, stream=None):
    """code_t(k_i) per key and table: int32 [B, Hkv, n, L]."""
    out = torch.empty(B, Hkv, n, L, dtype=torch.int32, device=codes.device)
    _check(lib().mp_codes_unpack(_ptr(codes), B, Hkv, n, K, L, _ptr(out), _stream(stream)),
           "mp_codes_unpack")
    return out


def device_status() -> int:
    """Synchronise the device; return and clear its status word (0 = MP_OK, 4 = timeout,
    6 = a failed index check of the MP_CHECKS build)."""
    v = _c_int(0)
    _check(lib().mp_device_status(ctypes.byref(v)), "mp_device_status")
    return int(v.value)


def check_report() -> tuple[bool, int]:
    """(whether the loaded library is the MP_CHECKS build, the site of the first failed index
    check since the status word was last cleared, 0 if none); clears nothing."""
    en, site = _c_int(0), _c_int(0)
    _check(lib().mp_debug_check_report(ctypes.byref(en), ctypes.byref(site)),
           "mp_debug_check_report")
    return bool(en.value), int(site.value)
