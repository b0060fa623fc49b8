"""Thin Python binding of libdendrite.so (argument marshalling only).

Every step of the path (fork, copy-on-write append, planning, attention,
merge, free) runs inside the C-ABI library and its CUDA kernels; this module
only turns torch tensors into device pointers and the current torch stream
into a ``cudaStream_t``.  If the library is missing it raises at import of
:func:`lib` -- there is no fallback.
"""
from __future__ import annotations

import array
import ctypes
import os
from typing import List, Optional, Sequence

import torch

from . import _build

__all__ = ["lib", "Pool", "DendriteError", "ERRORS", "plan_segments", "TIMING_NAMES"]

ERRORS = {
    -1: "EINVAL", -2: "ENOMEM", -3: "EBADHANDLE", -4: "ELIMIT", -5: "EDTYPE",
    -6: "ECUDA", -7: "ETIMEOUT", -8: "ECORRUPT",
}
TIMING_NAMES = ("fork", "append_meta", "append_copy", "attn_partial", "attn_merge", "free", "attn_total",
                "attn_tc", "attn_mma_side")
FP32, BF16, TURBO = 0, 1, 2
TURBO_KEY_BYTES, TURBO_VALUE_BYTES = 96, 64

_LIB = None
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_pi32 = ctypes.c_void_p


class DendriteError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        self.name = ERRORS.get(code, str(code))
        super().__init__(f"dendrite error {self.name} ({code}){': ' + what if what else ''}")


class _Opts(ctypes.Structure):
    _fields_ = [("max_branches", _i32), ("max_blocks_per_branch", _i32), ("tc_min_rows", _i32),
                ("n_layers", _i32), ("fold_segments", _i32), ("device_planning", _i32), ("tc_sms", _i32), ("pack_segments", _i32),
                ("reserved", _i32 * 1)]


class _PlanStats(ctypes.Structure):
    _fields_ = [("n_segments", _i32), ("n_units", _i32), ("n_ctas", _i32), ("n_partials", _i32),
                ("tiles", _i64), ("unique_tiles", _i64), ("plan_us", ctypes.c_double), ("n_tc_units", _i32),
                ("n_tc_ctas", _i32), ("refreshed", _i32), ("reserved", _i32)]


class _Segment(ctypes.Structure):
    _fields_ = [("rep", _i32), ("block_start", _i32), ("block_count", _i32),
                ("member_offset", _i32), ("n_members", _i32)]


class _ExtraTile(ctypes.Structure):
    _fields_ = [("rep", _i32), ("block", _i32), ("member_mask", ctypes.c_uint32), ("reserved", _i32)]


_SIGS = {
    "dendrite_pool_create": [_i64, _i32, _i32, _i32, _i32, ctypes.POINTER(_Opts), ctypes.POINTER(_p)],
    "dendrite_pool_create_turbo": [_i64, _i32, _i32, _i32, _p, _p, ctypes.POINTER(_Opts), ctypes.POINTER(_p)],
    "dendrite_pool_destroy": [_p],
    "dendrite_branch_new": [_p, _pi32],
    "dendrite_fork": [_p, _i32, _i32, _pi32, _p],
    "dendrite_fork_batch": [_p, _pi32, _pi32, _i32, _pi32, _p],
    "dendrite_append_kv": [_p, _pi32, _i32, _i32, _p, _p, _p],
    "dendrite_append_begin": [_p, _pi32, _i32, _i32, _p],
    "dendrite_append_layer": [_p, _i32, _p, _p, _p],
    "dendrite_tree_attn_decode_layer": [_p, _i32, _p, _i32, _i32, _pi32, _i32, _p, _p],
    "dendrite_read_block_layer": [_p, _i32, _i32, _p, _p, _p],
    "dendrite_pool_layers": [_p, _pi32],
    "dendrite_selftest_bounded_wait": [_p, _p],
    "dendrite_tree_attn_decode": [_p, _p, _i32, _i32, _pi32, _i32, _p, _p],
    "dendrite_tree_attn_decode_noalloc": [_p, _p, _i32, _i32, _pi32, _i32, _p, _p],
    "dendrite_free": [_p, _pi32, _i32, _p],
    "dendrite_truncate": [_p, _pi32, _pi32, _i32, _p],
    "dendrite_sync": [_p, _p],
    "dendrite_branch_len": [_p, _i32, _pi32],
    "dendrite_read_table": [_p, _i32, _pi32, _i32, _pi32, _p],
    "dendrite_read_refcounts": [_p, _pi32, _p],
    "dendrite_read_free_stack": [_p, _pi32, _pi32, _p],
    "dendrite_read_block": [_p, _i32, _p, _p, _p],
    "dendrite_pool_info": [_p, ctypes.POINTER(_i64), _pi32, _pi32, _pi32, _pi32],
    "dendrite_set_profiling": [_p, _i32],
    "dendrite_last_timings": [_p, ctypes.POINTER(ctypes.c_float), _i32],
    "dendrite_last_plan_stats": [_p, ctypes.POINTER(_PlanStats)],
    "dendrite_plan_segments": [_i32, _pi32, _pi32, _pi32, _i32, _pi32, _i32, ctypes.POINTER(_Segment), _i32,
                               _pi32, _pi32, _i32, _pi32],
    "dendrite_plan_segments_folded": [_i32, _pi32, _pi32, _pi32, _i32, _pi32, _i32, _i32, _i32, _i32,
                                      ctypes.POINTER(_Segment), _i32, _pi32, _pi32, _i32, _pi32],
    "dendrite_plan_segments_packed": [_i32, _pi32, _pi32, _pi32, _i32, _pi32, _i32, _i32, _i32, _i32, _i32,
                                      ctypes.POINTER(_Segment), _i32, _pi32, _pi32, _i32, _pi32, _pi32,
                                      ctypes.POINTER(_ExtraTile), _i32, _pi32],
}


def lib() -> ctypes.CDLL:
    """Load libdendrite.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.dendrite_version.restype = ctypes.c_char_p
        L.dendrite_version.argtypes = []
        _LIB = L
    return _LIB


def _check(rc: int, what: str = "") -> None:
    if rc != 0:
        raise DendriteError(rc, what)


def _arr(xs: Sequence[int]) -> array.array:
    """int32 host buffer (kept alive by the caller for the duration of the call)."""
    a = array.array("i", xs)
    if not a:
        a.append(0)
    return a


def _ptr(a: array.array) -> int:
    return a.buffer_info()[0]


try:
    _raw_stream = torch._C._cuda_getCurrentRawStream
except AttributeError:  # pragma: no cover
    _raw_stream = None


def _stream_ptr(stream, device_index: int = 0) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(device_index)
    return torch.cuda.current_stream().cuda_stream


_DT = {torch.float32: FP32, torch.bfloat16: BF16}


class Pool:
    """A device block pool with copy-on-write branch forking and tree decode attention."""

    def __init__(self, num_blocks: int, block_size: int = 16, n_kv_heads: int = 8, head_dim: int = 128,
                 dtype: torch.dtype = torch.bfloat16, max_branches: int = 4096,
                 max_blocks_per_branch: int = 4096, device=None, tc_min_rows: int = 0, n_layers: int = 1,
                 fold_segments: int = 0, turbo=None, device_planning: int = 0, tc_sms: int = 0,
                 pack_segments: int = 0):
        """``turbo``: (rotation signs [128], QJL matrix [128][128]) to store
        compressed blocks (dendrite_pool_create_turbo); the calls then take
        bf16 tensors."""
        if dtype not in _DT or (turbo is not None and dtype != torch.bfloat16):
            raise DendriteError(-5, f"dtype {dtype}")
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.n_kv_heads, self.head_dim, self.dtype = int(n_kv_heads), int(head_dim), dtype
        opts = _Opts(int(max_branches), int(max_blocks_per_branch), int(tc_min_rows), int(n_layers),
                     int(fold_segments), int(device_planning), int(tc_sms), int(pack_segments))
        self.n_layers = int(n_layers)
        self.turbo = turbo is not None
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            if self.turbo:
                signs = torch.as_tensor(turbo[0], dtype=torch.float32).contiguous().cpu()
                S = torch.as_tensor(turbo[1], dtype=torch.float32).contiguous().cpu()
                if signs.numel() != self.head_dim or S.shape != (128, self.head_dim):
                    raise DendriteError(-1, "turbo codec shapes")
                _check(lib().dendrite_pool_create_turbo(self.num_blocks, self.block_size, self.n_kv_heads,
                                                        self.head_dim, signs.data_ptr(), S.data_ptr(),
                                                        ctypes.byref(opts), ctypes.byref(h)), "pool_create_turbo")
            else:
                _check(lib().dendrite_pool_create(self.num_blocks, self.block_size, self.n_kv_heads, self.head_dim,
                                                  _DT[dtype], ctypes.byref(opts), ctypes.byref(h)), "pool_create")
        self._h = h
        self._dev = self.device.index

    # ------------------------------------------------------------ lifetime
    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().dendrite_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # --------------------------------------------------------------- ops
    def new_branch(self) -> int:
        out = ctypes.c_int32()
        _check(lib().dendrite_branch_new(self._h, ctypes.addressof(out)), "branch_new")
        return out.value

    def fork(self, parent: int, n_children: int, stream=None) -> List[int]:
        out = (ctypes.c_int32 * n_children)()
        _check(lib().dendrite_fork(self._h, int(parent), int(n_children), ctypes.addressof(out),
                                   _stream_ptr(stream, self._dev)),
               "fork")
        return list(out)

    def fork_batch(self, parents: Sequence[int], n_children: Sequence[int], stream=None) -> List[List[int]]:
        n_par = len(parents)
        pa, na = _arr(parents), _arr(n_children)
        total = sum(na) if n_par else 0
        out = array.array("i", bytes(4 * max(1, total)))
        _check(lib().dendrite_fork_batch(self._h, _ptr(pa), _ptr(na), n_par, _ptr(out),
                                         _stream_ptr(stream, self._dev)), "fork_batch")
        if n_par == 0:
            return []
        flat = out.tolist()
        if total == len(na):
            return [[x] for x in flat]
        res, k = [], 0
        for n in na:
            res.append(flat[k:k + n])
            k += n
        return res

    def fork_each(self, parents: Sequence[int], stream=None) -> List[int]:
        """One child per parent (dendrite_fork_batch with every count 1): the
        children's handles, in the parents' order."""
        n = len(parents)
        if n == 0:
            return []
        pa = _arr(parents)
        na = array.array("i", [1]) * n
        out = array.array("i", bytes(4 * n))
        _check(lib().dendrite_fork_batch(self._h, _ptr(pa), _ptr(na), n, _ptr(out),
                                         _stream_ptr(stream, self._dev)), "fork_each")
        return out.tolist()

    def _check_tensor(self, t: torch.Tensor, name: str) -> None:
        if not t.is_cuda or t.dtype != self.dtype or not t.is_contiguous():
            raise DendriteError(-1, f"{name} must be a contiguous {self.dtype} CUDA tensor")

    def append_kv(self, branches: Sequence[int], K: torch.Tensor, V: torch.Tensor, stream=None) -> None:
        """K, V: ``[n_branches][n_new][n_kv_heads][head_dim]``; for a pool of
        several layers ``[n_layers][n_branches][n_new][n_kv_heads][head_dim]``."""
        self._check_tensor(K, "K")
        self._check_tensor(V, "V")
        nb = len(branches)
        want = 4 if self.n_layers == 1 else 5
        if K.shape != V.shape or K.dim() != want or (want == 5 and K.shape[0] != self.n_layers):
            raise DendriteError(-1, f"K/V shape {tuple(K.shape)}")
        k4 = K.shape[-4:]
        if k4[0] != nb or k4[2] != self.n_kv_heads or k4[3] != self.head_dim:
            raise DendriteError(-1, f"K/V shape {tuple(K.shape)}")
        ba = _arr(branches)
        _check(lib().dendrite_append_kv(self._h, _ptr(ba), nb, k4[1], K.data_ptr(), V.data_ptr(),
                                        _stream_ptr(stream, self._dev)), "append_kv")

    def append_begin(self, branches: Sequence[int], n_new: int, stream=None) -> None:
        """Block decisions and new lengths of an append, for every layer; rows follow per layer."""
        ba = _arr(branches)
        _check(lib().dendrite_append_begin(self._h, _ptr(ba), len(branches), int(n_new),
                                           _stream_ptr(stream, self._dev)), "append_begin")

    def append_layer(self, layer: int, K: torch.Tensor, V: torch.Tensor, stream=None) -> None:
        """Rows of the pending append for one layer: K, V ``[n_branches][n_new][n_kv_heads][head_dim]``."""
        self._check_tensor(K, "K")
        self._check_tensor(V, "V")
        if K.shape != V.shape or K.dim() != 4 or K.shape[2] != self.n_kv_heads or K.shape[3] != self.head_dim:
            raise DendriteError(-1, f"K/V shape {tuple(K.shape)}")
        _check(lib().dendrite_append_layer(self._h, int(layer), K.data_ptr(), V.data_ptr(),
                                           _stream_ptr(stream, self._dev)), "append_layer")

    def tree_attn_decode(self, Q: torch.Tensor, branches: Sequence[int], out: Optional[torch.Tensor] = None,
                         stream=None, layer: int = 0) -> torch.Tensor:
        """Q: ``[n_branches][q_len][n_q_heads][head_dim]``; returns out of the same shape."""
        self._check_tensor(Q, "Q")
        if Q.dim() != 4 or Q.shape[0] != len(branches) or Q.shape[3] != self.head_dim:
            raise DendriteError(-1, f"Q shape {tuple(Q.shape)}")
        if out is None:
            out = torch.empty_like(Q)
        self._check_tensor(out, "out")
        if out.shape != Q.shape:
            raise DendriteError(-1, "out shape")
        ba = _arr(branches)
        _check(lib().dendrite_tree_attn_decode_layer(self._h, int(layer), Q.data_ptr(), Q.shape[2], Q.shape[1],
                                                     _ptr(ba), len(branches), out.data_ptr(),
                                                     _stream_ptr(stream, self._dev)),
               "tree_attn_decode")
        return out

    def tree_attn_decode_noalloc(self, Q: torch.Tensor, branches: Sequence[int], out: torch.Tensor,
                                 stream=None) -> torch.Tensor:
        """Same as :meth:`tree_attn_decode` but with scratch in the library's fixed
        16 MiB per-device array (no device allocation during the call); ``out``
        must be given.  Raises ELIMIT when the plan and partials do not fit."""
        self._check_tensor(Q, "Q")
        self._check_tensor(out, "out")
        if Q.dim() != 4 or Q.shape[0] != len(branches) or Q.shape[3] != self.head_dim or out.shape != Q.shape:
            raise DendriteError(-1, f"Q/out shape {tuple(Q.shape)}")
        ba = _arr(branches)
        _check(lib().dendrite_tree_attn_decode_noalloc(self._h, Q.data_ptr(), Q.shape[2], Q.shape[1], _ptr(ba),
                                                       len(branches), out.data_ptr(),
                                                       _stream_ptr(stream, self._dev)),
               "tree_attn_decode_noalloc (scratch limit 16 MiB)")
        return out

    def free(self, branches: Sequence[int], stream=None) -> None:
        ba = _arr(branches)
        _check(lib().dendrite_free(self._h, _ptr(ba), len(branches), _stream_ptr(stream, self._dev)), "free")

    def truncate(self, branches: Sequence[int], new_lens: Sequence[int], stream=None) -> None:
        """Roll branch i back to its first ``new_lens[i]`` tokens."""
        ba, la = _arr(branches), _arr(new_lens)
        if len(branches) != len(new_lens):
            raise DendriteError(-1, "branches / new_lens length")
        _check(lib().dendrite_truncate(self._h, _ptr(ba), _ptr(la), len(branches), _stream_ptr(stream, self._dev)),
               "truncate")

    def sync(self, stream=None) -> None:
        _check(lib().dendrite_sync(self._h, _stream_ptr(stream, self._dev)), "sync")

    def sync_status(self, stream=None) -> int:
        """Like :meth:`sync` but returns the status code instead of raising."""
        return lib().dendrite_sync(self._h, _stream_ptr(stream, self._dev))

    # -------------------------------------------------------- inspection
    def branch_len(self, b: int) -> int:
        out = ctypes.c_int32()
        _check(lib().dendrite_branch_len(self._h, int(b), ctypes.addressof(out)), "branch_len")
        return out.value

    def read_table(self, b: int, stream=None) -> List[int]:
        n = ctypes.c_int32()
        cap = (self.branch_len(b) + self.block_size - 1) // self.block_size
        buf = (ctypes.c_int32 * max(1, cap))()
        _check(lib().dendrite_read_table(self._h, int(b), ctypes.addressof(buf), cap, ctypes.addressof(n),
                                         _stream_ptr(stream, self._dev)),
               "read_table")
        return list(buf[:n.value])

    def read_refcounts(self, stream=None) -> List[int]:
        buf = (ctypes.c_int32 * self.num_blocks)()
        _check(lib().dendrite_read_refcounts(self._h, ctypes.addressof(buf), _stream_ptr(stream, self._dev)),
               "read_refcounts")
        return list(buf)

    def read_free_stack(self, stream=None) -> List[int]:
        buf = (ctypes.c_int32 * self.num_blocks)()
        top = ctypes.c_int32()
        _check(lib().dendrite_read_free_stack(self._h, ctypes.addressof(buf), ctypes.addressof(top),
                                              _stream_ptr(stream, self._dev)),
               "read_free_stack")
        return list(buf[:top.value])

    def read_block(self, blk: int, stream=None, layer: int = 0):
        """K and V of a block: [n_kv_heads][block_size][head_dim] in the pool
        dtype, or the raw records ([...][96] and [...][64] uint8) of a
        compressed pool."""
        if self.turbo:
            k = torch.empty((self.n_kv_heads, self.block_size, TURBO_KEY_BYTES), dtype=torch.uint8)
            v = torch.empty((self.n_kv_heads, self.block_size, TURBO_VALUE_BYTES), dtype=torch.uint8)
        else:
            shape = (self.n_kv_heads, self.block_size, self.head_dim)
            k = torch.empty(shape, dtype=self.dtype)
            v = torch.empty(shape, dtype=self.dtype)
        _check(lib().dendrite_read_block_layer(self._h, int(layer), int(blk), k.data_ptr(), v.data_ptr(),
                                               _stream_ptr(stream, self._dev)), "read_block")
        return k, v

    # --------------------------------------------------------- profiling
    def set_profiling(self, enable) -> None:
        """True/1: events around every kernel; 2: around whole attention calls only."""
        level = 2 if enable == 2 else (1 if enable else 0)
        _check(lib().dendrite_set_profiling(self._h, level), "set_profiling")

    def last_timings(self) -> dict:
        buf = (ctypes.c_float * len(TIMING_NAMES))()
        _check(lib().dendrite_last_timings(self._h, buf, len(TIMING_NAMES)), "last_timings")
        return {k: (v if v >= 0 else None) for k, v in zip(TIMING_NAMES, buf)}

    def last_plan_stats(self) -> dict:
        st = _PlanStats()
        _check(lib().dendrite_last_plan_stats(self._h, ctypes.byref(st)), "last_plan_stats")
        return {f: getattr(st, f) for f, _ in _PlanStats._fields_}


def plan_segments(parent: Sequence[int], fork_len: Sequence[int], length: Sequence[int], block_size: int,
                  queried: Sequence[int], rows_per_member: int = 0, tc_min_rows: int = 0, fold_pct: int = 0):
    """Host planner (no GPU): returns a list of (rep, block_start, block_count, members).
    rows_per_member > 0: the folded segments the bf16 attention call reads
    (dendrite_plan_segments_folded), else the maximal sharing segments."""
    n = len(parent)
    ns, nm = ctypes.c_int32(), ctypes.c_int32()
    L = lib()
    pa, fa, la, qa = _arr(parent), _arr(fork_len), _arr(length), _arr(queried)
    head = (n, _ptr(pa), _ptr(fa), _ptr(la), block_size, _ptr(qa), len(queried))
    if rows_per_member > 0:
        fn, name = L.dendrite_plan_segments_folded, "plan_segments_folded"
        head = head + (int(rows_per_member), int(tc_min_rows), int(fold_pct))
    else:
        fn, name = L.dendrite_plan_segments, "plan_segments"
    rc = fn(*head, None, 0, ctypes.addressof(ns), None, 0, ctypes.addressof(nm))
    if rc not in (0, -4):
        _check(rc, name)
    segs = (_Segment * max(1, ns.value))()
    mem = (ctypes.c_int32 * max(1, nm.value))()
    _check(fn(*head, segs, ns.value, ctypes.addressof(ns), ctypes.addressof(mem), nm.value, ctypes.addressof(nm)),
           name)
    out = []
    for s in segs[:ns.value]:
        out.append((s.rep, s.block_start, s.block_count, list(mem[s.member_offset:s.member_offset + s.n_members])))
    return out


def plan_segments_packed(parent: Sequence[int], fork_len: Sequence[int], length: Sequence[int], block_size: int,
                         queried: Sequence[int], rows_per_member: int, tc_min_rows: int = 0, fold_pct: int = 0,
                         pack_pct: int = 0):
    """Host planner with packing, then folding (dendrite_plan_segments_packed):
    a list of (rep, block_start, block_count, members, extras), extras being
    (rep, block, member_mask) tuples."""
    n = len(parent)
    ns, nm, nx = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    L = lib()
    pa, fa, la, qa = _arr(parent), _arr(fork_len), _arr(length), _arr(queried)
    head = (n, _ptr(pa), _ptr(fa), _ptr(la), block_size, _ptr(qa), len(queried), int(rows_per_member),
            int(tc_min_rows), int(fold_pct), int(pack_pct))
    fn = L.dendrite_plan_segments_packed
    rc = fn(*head, None, 0, ctypes.addressof(ns), None, 0, ctypes.addressof(nm), None, None, 0,
            ctypes.addressof(nx))
    if rc not in (0, -4):
        _check(rc, "plan_segments_packed")
    segs = (_Segment * max(1, ns.value))()
    mem = (ctypes.c_int32 * max(1, nm.value))()
    xo = (ctypes.c_int32 * (ns.value + 1))()
    xt = (_ExtraTile * max(1, nx.value))()
    _check(fn(*head, segs, ns.value, ctypes.addressof(ns), ctypes.addressof(mem), nm.value, ctypes.addressof(nm),
              ctypes.addressof(xo), xt, nx.value, ctypes.addressof(nx)), "plan_segments_packed")
    out = []
    for k, s in enumerate(segs[:ns.value]):
        ex = [(e.rep, e.block, e.member_mask) for e in xt[xo[k]:xo[k + 1]]]
        out.append((s.rep, s.block_start, s.block_count, list(mem[s.member_offset:s.member_offset + s.n_members]),
                    ex))
    return out
