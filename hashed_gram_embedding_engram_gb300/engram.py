"""Python front end of the Engram C ABI: argument marshalling only.

Every step of the layer runs in the library's CUDA kernels (libengram_gb300.so);
torch provides device memory and the current stream.  Tensors are passed by
pointer; no tensor is copied or converted here except where a method says so
(``EngramLayer.__call__`` moves host inputs to the device and back).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence, Tuple

import torch

from . import _lib

_TABLE_DTYPES = {"f32": (_lib.F32, torch.float32), "bf16": (_lib.BF16, torch.bfloat16),
                 "i8": (_lib.I8_ROWSCALE_F16, torch.int8)}
_ACT_DTYPES = {"f32": (_lib.F32, torch.float32), "bf16": (_lib.BF16, torch.bfloat16)}


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _dev_or_pinned(t: torch.Tensor, name: str, dtype) -> int:
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name}: host tables must be pinned (read by the GPU over UVA)")
    return t.data_ptr()


@dataclass
class EngramWeights:
    """One layer's parameters (see engram_weights_t).  ``table`` / ``scales`` may be
    pinned host tensors; everything else lives on the device."""
    table: torch.Tensor            # [sum primes, row_dim]
    w_kv: torch.Tensor             # [(M+1)d, d_mem]: W_V then W_K^(1..M)
    g_h: torch.Tensor              # float32 [M, d]
    g_k: torch.Tensor              # float32 [M, d]
    g_c: torch.Tensor              # float32 [d]
    conv: torch.Tensor             # float32 [d, w]
    scales: Optional[torch.Tensor] = None   # float16 [sum primes] for int8 tables
    # FP8 projection: W_kv as e4m3 codes [(M+1)d, d_mem] (uint8) with float32
    # row scales [(M+1)d], from EngramPlan.quantize_fp8(w_kv); w_kv is then unused
    w_kv_fp8: Optional[torch.Tensor] = None
    w_kv_scale: Optional[torch.Tensor] = None

    def struct(self, plan: "EngramPlan", need_table: bool = True) -> _lib.Weights:
        c = plan
        tdt = _TABLE_DTYPES[c.table_dtype][1]
        adt = _ACT_DTYPES[c.act_dtype][1]
        w = _lib.Weights()
        if need_table:
            w.table = _dev_or_pinned(self.table, "table", tdt)
            if self.table.shape != (c.total_rows, c.row_dim):
                raise ValueError(f"table: shape {tuple(self.table.shape)}, expected {(c.total_rows, c.row_dim)}")
            if c.table_dtype == "i8":
                if self.scales is None:
                    raise ValueError("int8 tables need fp16 row scales")
                w.scales = _dev_or_pinned(self.scales, "scales", torch.float16)
        if self.w_kv_fp8 is not None:
            w.w_kv_fp8 = _dev(self.w_kv_fp8, "w_kv_fp8", torch.uint8, ((c.M + 1) * c.d, c.d_mem))
            w.w_kv_scale = _dev(self.w_kv_scale, "w_kv_scale", torch.float32, ((c.M + 1) * c.d,))
        if self.w_kv is not None:
            w.w_kv = _dev(self.w_kv, "w_kv", adt, ((c.M + 1) * c.d, c.d_mem))
        w.g_h = _dev(self.g_h, "g_h", torch.float32, (c.M, c.d))
        w.g_k = _dev(self.g_k, "g_k", torch.float32, (c.M, c.d))
        w.g_c = _dev(self.g_c, "g_c", torch.float32, (c.d,))
        w.conv = _dev(self.conv, "conv", torch.float32, (c.d, c.conv_w))
        return w


@dataclass
class EngramState:
    """Streaming state of B sequences (see engram_state_t); zeros = fresh."""
    prev_ids: torch.Tensor         # int32 [B, N-1]
    u_ring: torch.Tensor           # float32 [B, L, M, d]
    pos: torch.Tensor              # int32 [B]

    @classmethod
    def zeros(cls, plan: "EngramPlan", B: int, device="cuda") -> "EngramState":
        L = max(1, (plan.conv_w - 1) * plan.conv_dilation)
        return cls(torch.zeros(B, plan.N - 1, dtype=torch.int32, device=device),
                   torch.zeros(B, L, plan.M, plan.d, dtype=torch.float32, device=device),
                   torch.zeros(B, dtype=torch.int32, device=device))

    def struct(self, plan: "EngramPlan", B: int) -> _lib.State:
        L = max(1, (plan.conv_w - 1) * plan.conv_dilation)
        s = _lib.State()
        s.prev_ids = _dev(self.prev_ids, "prev_ids", torch.int32, (B, plan.N - 1))
        s.u_ring = _dev(self.u_ring, "u_ring", torch.float32, (B, L, plan.M, plan.d))
        s.pos = _dev(self.pos, "pos", torch.int32, (B,))
        return s

    def clone(self) -> "EngramState":
        return EngramState(self.prev_ids.clone(), self.u_ring.clone(), self.pos.clone())

    def rows(self, lo: int, hi: int) -> "EngramState":
        """The state of sequences lo..hi-1 (views: updates land in this state)."""
        return EngramState(self.prev_ids[lo:hi], self.u_ring[lo:hi], self.pos[lo:hi])


class EngramPlan:
    """A validated layer configuration bound to the current CUDA device."""

    def __init__(self, *, N: int, K: int, row_dim: int, d: int, M: int = 1, conv_w: int = 4,
                 conv_dilation: Optional[int] = None, table_dtype: str = "bf16", act_dtype: str = "bf16",
                 eps: float = 1e-6, primes: Sequence[int], multipliers: Sequence[int], max_tokens: int):
        self.N, self.K, self.row_dim, self.d, self.M = N, K, row_dim, d, M
        self.conv_w = conv_w
        self.conv_dilation = N if conv_dilation is None else conv_dilation
        self.table_dtype, self.act_dtype, self.eps = table_dtype, act_dtype, eps
        self.R = (N - 1) * K
        self.d_mem = self.R * row_dim
        self.primes = [int(p) for p in primes]
        self.total_rows = sum(self.primes)
        self.max_tokens = int(max_tokens)
        if len(self.primes) != self.R:
            raise ValueError(f"need {self.R} primes, got {len(self.primes)}")
        n_mult = sum(K * n for n in range(2, N + 1))
        mults = [int(m) for m in multipliers]
        if len(mults) != n_mult:
            raise ValueError(f"need {n_mult} multipliers, got {len(mults)}")
        self._primes_c = (ctypes.c_uint32 * self.R)(*self.primes)
        self._mults_c = (ctypes.c_uint64 * n_mult)(*mults)
        cfg = _lib.Config(N, K, row_dim, d, M, conv_w, self.conv_dilation, _TABLE_DTYPES[table_dtype][0],
                          _ACT_DTYPES[act_dtype][0], eps, self._primes_c, self._mults_c)
        self._lib = _lib._lib()
        self._h = ctypes.c_void_p()
        torch.cuda.current_device()   # make sure a context exists on the current device
        _lib.check(self._lib.engram_plan_create(ctypes.byref(cfg), self.max_tokens, ctypes.byref(self._h)),
                   "engram_plan_create")

    # ------------------------------------------------------------ helpers
    @property
    def act_torch_dtype(self) -> torch.dtype:
        return _ACT_DTYPES[self.act_dtype][1]

    def workspace_bytes(self, ntok: int) -> int:
        n = ctypes.c_size_t()
        _lib.check(self._lib.engram_plan_workspace_bytes(self._h, ntok, ctypes.byref(n)), "workspace_bytes")
        return n.value

    def new_workspace(self, ntok: int, device="cuda") -> torch.Tensor:
        return torch.empty(max(1, self.workspace_bytes(ntok)), dtype=torch.uint8, device=device)

    def close(self) -> None:
        if getattr(self, "_h", None) and self._h.value:
            self._lib.engram_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ entry points
    def hash(self, ids: torch.Tensor, proj: torch.Tensor, prev_ids: Optional[torch.Tensor] = None,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Steps 1-3: int32 ids [B, T] -> int32 indices [B*T, R]."""
        B, T = ids.shape
        if out is None:
            out = torch.empty(B * T, self.R, dtype=torch.int32, device=ids.device)
        prev = 0 if prev_ids is None else _dev(prev_ids, "prev_ids", torch.int32, (B, self.N - 1))
        _lib.check(self._lib.engram_hash(self._h, _dev(ids, "ids", torch.int32), B, T,
                                         _dev(proj, "proj", torch.int32), proj.numel(), prev,
                                         _dev(out, "idx_out", torch.int32, (B * T, self.R)), _stream()),
                   "engram_hash")
        return out

    def gather(self, idx: torch.Tensor, table: torch.Tensor, scales: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Step 4: int32 indices [ntok, R] -> e [ntok, d_mem] (act dtype)."""
        ntok = idx.shape[0]
        if out is None:
            out = torch.empty(ntok, self.d_mem, dtype=self.act_torch_dtype, device=idx.device)
        tab = _dev_or_pinned(table, "table", _TABLE_DTYPES[self.table_dtype][1])
        sc = 0 if scales is None else _dev_or_pinned(scales, "scales", torch.float16)
        _lib.check(self._lib.engram_gather(self._h, _dev(idx, "idx", torch.int32, (ntok, self.R)), ntok, tab, sc,
                                           _dev(out, "e_out", self.act_torch_dtype, (ntok, self.d_mem)), _stream()),
                   "engram_gather")
        return out

    def stage_a(self, ids: torch.Tensor, proj: torch.Tensor, table: torch.Tensor,
                scales: Optional[torch.Tensor] = None, prev_ids: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Steps 1-4 in one kernel: int32 ids [B, T] -> e [B*T, d_mem] (act dtype)."""
        B, T = ids.shape
        if out is None:
            out = torch.empty(B * T, self.d_mem, dtype=self.act_torch_dtype, device=ids.device)
        prev = 0 if prev_ids is None else _dev(prev_ids, "prev_ids", torch.int32, (B, self.N - 1))
        tab = _dev_or_pinned(table, "table", _TABLE_DTYPES[self.table_dtype][1])
        sc = 0 if scales is None else _dev_or_pinned(scales, "scales", torch.float16)
        _lib.check(self._lib.engram_stage_a(self._h, _dev(ids, "ids", torch.int32), B, T,
                                            _dev(proj, "proj", torch.int32), proj.numel(), prev, tab, sc,
                                            _dev(out, "e_out", self.act_torch_dtype, (B * T, self.d_mem)),
                                            _stream()), "engram_stage_a")
        return out

    def quantize_fp8(self, x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
        """Per-row e4m3 codes (uint8, same shape) and float32 scales of a bf16
        [rows, cols] device tensor (engram_quantize_fp8)."""
        if x.dim() != 2:
            raise ValueError("x: expected a 2-D tensor")
        rows, cols = x.shape
        q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device)
        sc = torch.empty(rows, dtype=torch.float32, device=x.device)
        _lib.check(self._lib.engram_quantize_fp8(self._h, _dev(x, "x", torch.bfloat16), rows, cols, _dev(q, "q"),
                                                 _dev(sc, "scale"), _stream()), "engram_quantize_fp8")
        return q, sc

    def kv_projection(self, e: torch.Tensor, w_kv: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Step 5: e [ntok, d_mem] -> kv [ntok, (M+1)d] = e . w_kv^T."""
        ntok = e.shape[0]
        nc = (self.M + 1) * self.d
        if out is None:
            out = torch.empty(ntok, nc, dtype=self.act_torch_dtype, device=e.device)
        _lib.check(self._lib.engram_kv_projection(
            self._h, _dev(e, "e", self.act_torch_dtype, (ntok, self.d_mem)), ntok,
            _dev(w_kv, "w_kv", self.act_torch_dtype, (nc, self.d_mem)),
            _dev(out, "kv_out", self.act_torch_dtype, (ntok, nc)), _stream()), "engram_kv_projection")
        return out

    def stage_b(self, e: torch.Tensor, weights: EngramWeights, H: torch.Tensor, state: Optional[EngramState] = None,
                ids: Optional[torch.Tensor] = None, proj: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Steps 5-8 in place on H [B, T, M, d] from gathered rows e [B*T, d_mem].

        With a ``state``, ``ids`` [B, T] and ``proj`` are needed too."""
        B, T = H.shape[0], H.shape[1]
        ws = self.new_workspace(B * T, H.device) if workspace is None else workspace
        w = weights.struct(self, need_table=False)
        st = None if state is None else ctypes.byref(state.struct(self, B))
        ids_p = 0 if ids is None else _dev(ids, "ids", torch.int32, (B, T))
        proj_p, V = (0, 0) if proj is None else (_dev(proj, "proj", torch.int32), proj.numel())
        _lib.check(self._lib.engram_stage_b(
            self._h, ids_p, B, T, proj_p, V, _dev(e, "e", self.act_torch_dtype, (B * T, self.d_mem)),
            ctypes.byref(w), _dev(H, "H", self.act_torch_dtype, (B, T, self.M, self.d)), st,
            _dev(ws, "workspace"), ws.numel(), _stream()), "engram_stage_b")
        return H

    def stage_a_e4m3(self, ids: torch.Tensor, proj: torch.Tensor, table: torch.Tensor,
                     prev_ids: Optional[torch.Tensor] = None,
                     out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
        """Steps 1-4 writing e's e4m3 codes [B*T, d_mem] and scales [B*T] instead of e
        (engram_stage_a_e4m3; bf16 layers)."""
        return stage_a_layers_e4m3([self], ids, proj, [table], None if prev_ids is None else [prev_ids],
                                   None if out is None else [out])[0]

    def stage_b_e4m3(self, e8: torch.Tensor, e_scale: torch.Tensor, weights: EngramWeights, H: torch.Tensor,
                     state: Optional[EngramState] = None, ids: Optional[torch.Tensor] = None,
                     proj: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Steps 5-8 from e's e4m3 codes and scales (engram_stage_b_e4m3); the weights carry W_kv in e4m3."""
        B, T = H.shape[0], H.shape[1]
        ws = self.new_workspace(B * T, H.device) if workspace is None else workspace
        w = weights.struct(self, need_table=False)
        st = None if state is None else ctypes.byref(state.struct(self, B))
        ids_p = 0 if ids is None else _dev(ids, "ids", torch.int32, (B, T))
        proj_p, V = (0, 0) if proj is None else (_dev(proj, "proj", torch.int32), proj.numel())
        _lib.check(self._lib.engram_stage_b_e4m3(
            self._h, ids_p, B, T, proj_p, V, _dev(e8, "e8", torch.uint8, (B * T, self.d_mem)),
            _dev(e_scale, "e_scale", torch.float32, (B * T,)), ctypes.byref(w),
            _dev(H, "H", self.act_torch_dtype, (B, T, self.M, self.d)), st, _dev(ws, "workspace"), ws.numel(),
            _stream()), "engram_stage_b_e4m3")
        return H

    def forward(self, ids: torch.Tensor, proj: torch.Tensor, weights: EngramWeights, H: torch.Tensor,
                state: Optional[EngramState] = None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
        """Steps 1-8 in place on H [B, T, M, d]; ``state`` continues sequences."""
        B, T = ids.shape
        ws = self.new_workspace(B * T, H.device) if workspace is None else workspace
        w = weights.struct(self)
        st = None if state is None else ctypes.byref(state.struct(self, B))
        _lib.check(self._lib.engram_forward(
            self._h, _dev(ids, "ids", torch.int32), B, T, _dev(proj, "proj", torch.int32), proj.numel(),
            ctypes.byref(w), _dev(H, "H", self.act_torch_dtype, (B, T, self.M, self.d)), st,
            _dev(ws, "workspace"), ws.numel(), _stream()), "engram_forward")
        return H

    def forward_split(self, split: "SmSplit", n_pieces: int, ids: torch.Tensor, proj: torch.Tensor,
                      weights: EngramWeights, H: torch.Tensor, state: Optional[EngramState] = None,
                      workspace: Optional[torch.Tensor] = None, cache: Optional["EngramCache"] = None) -> torch.Tensor:
        """``forward`` in ``n_pieces`` pieces of whole sequences on an SM split: each
        piece's Stage A on group 0 (through ``cache`` if given), its Stage B on
        group 1 once its rows are in (engram_forward_split); the same bits as
        ``forward``."""
        B, T = ids.shape
        ws = self.new_workspace(B * T, H.device) if workspace is None else workspace
        w = weights.struct(self)
        st = None if state is None else ctypes.byref(state.struct(self, B))
        _lib.check(self._lib.engram_forward_split(
            self._h, split._h, int(n_pieces), None if cache is None else cache._h, _dev(ids, "ids", torch.int32), B, T,
            _dev(proj, "proj", torch.int32),
            proj.numel(), ctypes.byref(w), _dev(H, "H", self.act_torch_dtype, (B, T, self.M, self.d)), st,
            _dev(ws, "workspace"), ws.numel(), _stream()), "engram_forward_split")
        return H

    def set_fused_stage_b(self, enable: bool) -> None:
        """Stage B as one cooperative launch, or as two launches (the default); same bits."""
        _lib.check(self._lib.engram_plan_set_fused_stage_b(self._h, int(bool(enable))),
                   "engram_plan_set_fused_stage_b")

    def set_fused_decode(self, enable: bool) -> None:
        """Chunks of one position as one cooperative launch, or as separate launches (default); same bits."""
        _lib.check(self._lib.engram_plan_set_fused_decode(self._h, int(bool(enable))), "engram_plan_set_fused_decode")

    def set_cta_pairs(self, enable: bool) -> None:
        """The K/V projection's 256-column tiles on CTA pairs (cta_group::2), or one SM each; same bits."""
        _lib.check(self._lib.engram_plan_set_cta_pairs(self._h, int(bool(enable))), "engram_plan_set_cta_pairs")

    def set_sm_limit(self, n_sms: int) -> None:
        """At most n_sms SMs for Stage B's persistent kernels (0: all); the results do not depend on it."""
        _lib.check(self._lib.engram_plan_set_sm_limit(self._h, int(n_sms)), "engram_plan_set_sm_limit")

    def host_gather_sms(self) -> int:
        """SMs a Stage A over tables in pinned host memory occupies."""
        return int(self._lib.engram_plan_host_gather_sms(self._h))

    def set_host_gather_sms(self, n_sms: int) -> None:
        """SMs a Stage A over tables in pinned host memory runs on (0: a quarter of them); same bits."""
        _lib.check(self._lib.engram_plan_set_host_gather_sms(self._h, int(n_sms)), "engram_plan_set_host_gather_sms")

    def set_timing(self, enable: bool) -> None:
        """Record CUDA events around each kernel of later forward / stage_b calls."""
        _lib.check(self._lib.engram_plan_set_timing(self._h, int(bool(enable))), "engram_plan_set_timing")

    def kernel_times(self) -> list:
        """Device milliseconds of each kernel of the last call (waits for it)."""
        buf = (ctypes.c_float * 8)()
        n = ctypes.c_int()
        _lib.check(self._lib.engram_plan_kernel_times(self._h, buf, 8, ctypes.byref(n)), "engram_plan_kernel_times")
        return [buf[i] for i in range(n.value)]

    def get_error(self) -> Tuple[int, int]:
        """Synchronise the current stream; return (status, raw flag bits) and clear them."""
        flags = ctypes.c_uint32()
        st = self._lib.engram_get_error(self._h, _stream(), ctypes.byref(flags))
        return st, flags.value


class SmSplit:
    """The device's SMs in two disjoint sets, each with one stream whose kernels
    run on that set only (engram_sm_split_* in include/engram.h).  Group 0 has
    at least ``n_sms`` SMs (rounded up by the driver), group 1 the rest;
    ``stream(g)`` is a torch stream over group g's stream."""

    def __init__(self, n_sms: int, device: Optional[int] = None):
        self._lib = _lib._lib()
        dev = torch.cuda.current_device() if device is None else int(device)
        h = ctypes.c_void_p()
        _lib.check(self._lib.engram_sm_split_create(dev, int(n_sms), ctypes.byref(h)), "engram_sm_split_create")
        self._h = h
        self.device = dev
        self.sms = tuple(int(self._lib.engram_sm_split_sms(h, g)) for g in (0, 1))
        self._streams = tuple(torch.cuda.ExternalStream(int(self._lib.engram_sm_split_stream(h, g)), device=dev)
                              for g in (0, 1))

    def stream(self, group: int) -> torch.cuda.Stream:
        return self._streams[group]

    def close(self) -> None:
        """Destroys both streams: call after the work on them has completed."""
        if getattr(self, "_h", None):
            torch.cuda.synchronize(self.device)
            self._streams = ()
            _lib.check(self._lib.engram_sm_split_destroy(self._h), "engram_sm_split_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class EngramCache:
    """HBM hot-row cache in front of a host-resident table (engram_cache_* in
    include/engram.h): observe batches, build (LFU admission), then
    ``stage_a`` reads cached rows from HBM and the others over the host link."""

    def __init__(self, plan: "EngramPlan", capacity: int, table: torch.Tensor):
        self.plan = plan
        self._lib = _lib._lib()
        self._table = table                      # kept alive: the cache reads it
        tab = _dev_or_pinned(table, "table", _TABLE_DTYPES[plan.table_dtype][1])
        h = ctypes.c_void_p()
        _lib.check(self._lib.engram_cache_create(plan._h, int(capacity), tab, ctypes.byref(h)), "engram_cache_create")
        self._h = h

    def close(self) -> None:
        if getattr(self, "_h", None):
            _lib.check(self._lib.engram_cache_destroy(self._h), "engram_cache_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def observe(self, ids: torch.Tensor, proj: torch.Tensor, prev_ids: Optional[torch.Tensor] = None) -> None:
        B, T = ids.shape
        prev = 0 if prev_ids is None else _dev(prev_ids, "prev_ids", torch.int32, (B, self.plan.N - 1))
        _lib.check(self._lib.engram_cache_observe(self._h, _dev(ids, "ids", torch.int32), B, T,
                                                  _dev(proj, "proj", torch.int32), proj.numel(), prev, _stream()),
                   "engram_cache_observe")

    def build(self, decay: bool = False) -> int:
        n = ctypes.c_int64()
        _lib.check(self._lib.engram_cache_build(self._h, int(bool(decay)), _stream(), ctypes.byref(n)),
                   "engram_cache_build")
        return n.value

    def stage_a(self, ids: torch.Tensor, proj: torch.Tensor, scales: Optional[torch.Tensor] = None,
                prev_ids: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        plan = self.plan
        B, T = ids.shape
        if out is None:
            out = torch.empty(B * T, plan.d_mem, dtype=plan.act_torch_dtype, device=ids.device)
        prev = 0 if prev_ids is None else _dev(prev_ids, "prev_ids", torch.int32, (B, plan.N - 1))
        sc = 0 if scales is None else _dev_or_pinned(scales, "scales", torch.float16)
        _lib.check(self._lib.engram_stage_a_cached(self._h, _dev(ids, "ids", torch.int32), B, T,
                                                   _dev(proj, "proj", torch.int32), proj.numel(), prev, sc,
                                                   _dev(out, "e_out", plan.act_torch_dtype, (B * T, plan.d_mem)),
                                                   _stream()), "engram_stage_a_cached")
        return out

    def set_dedup(self, batch_rows: int) -> None:
        """Per-batch row dedup in ``stage_a``: each distinct uncached row of a
        batch crosses the host link once (room for ``batch_rows`` of them; 0 = off)."""
        _lib.check(self._lib.engram_cache_set_dedup(self._h, int(batch_rows)), "engram_cache_set_dedup")

    def stats(self, reset: bool = False) -> Tuple[int, int, int, int]:
        """(rows looked up, lookups served from HBM, rows read over the host link,
        rows cached) since the last reset."""
        a, b, l, c = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_int64()
        _lib.check(self._lib.engram_cache_stats(self._h, _stream(), int(bool(reset)), ctypes.byref(a), ctypes.byref(b),
                                                ctypes.byref(l), ctypes.byref(c)), "engram_cache_stats")
        return a.value, b.value, l.value, c.value


_COPY_STREAMS = {}


def stage_a_layers(plans: Sequence["EngramPlan"], ids: torch.Tensor, proj: torch.Tensor,
                   tables: Sequence[torch.Tensor], scales: Optional[Sequence[torch.Tensor]] = None,
                   prev_ids: Optional[Sequence[Optional[torch.Tensor]]] = None,
                   outs: Optional[Sequence[torch.Tensor]] = None) -> list:
    """Stage A of several layers of one shape in one launch (engram_stage_a_layers):
    int32 ids [B, T] -> one e [B*T, d_mem] per plan, the bits of per-layer stage_a."""
    n = len(plans)
    if n == 0 or len(tables) != n or (scales is not None and len(scales) != n) or \
            (prev_ids is not None and len(prev_ids) != n) or (outs is not None and len(outs) != n):
        raise ValueError("stage_a_layers: plans, tables, scales, prev_ids and outs must have one entry per layer")
    B, T = ids.shape
    p0 = plans[0]
    if outs is None:
        outs = [torch.empty(B * T, p.d_mem, dtype=p.act_torch_dtype, device=ids.device) for p in plans]
    arr = lambda vals: (ctypes.c_void_p * n)(*vals)  # noqa: E731
    h = arr([p._h.value for p in plans])
    tab = arr([_dev_or_pinned(t, "table", _TABLE_DTYPES[p.table_dtype][1]) for p, t in zip(plans, tables)])
    sc = 0 if scales is None else arr([_dev_or_pinned(s, "scales", torch.float16) for s in scales])
    prev = 0 if prev_ids is None else arr(
        [0 if x is None else _dev(x, "prev_ids", torch.int32, (B, p.N - 1)) for p, x in zip(plans, prev_ids)])
    out = arr([_dev(o, "e_out", p.act_torch_dtype, (B * T, p.d_mem)) for p, o in zip(plans, outs)])
    _lib.check(p0._lib.engram_stage_a_layers(n, h, _dev(ids, "ids", torch.int32), B, T,
                                             _dev(proj, "proj", torch.int32), proj.numel(), prev, tab, sc, out,
                                             _stream()), "engram_stage_a_layers")
    return list(outs)


def stage_a_layers_e4m3(plans: Sequence["EngramPlan"], ids: torch.Tensor, proj: torch.Tensor,
                        tables: Sequence[torch.Tensor], prev_ids: Optional[Sequence[Optional[torch.Tensor]]] = None,
                        outs: Optional[Sequence[Tuple[torch.Tensor, torch.Tensor]]] = None) -> list:
    """Stage A of several bf16 layers in one launch, writing each layer's e4m3
    codes [B*T, d_mem] (uint8) and per-token scales [B*T] (float32) instead of e
    (engram_stage_a_layers_e4m3): the bytes quantize_fp8 makes of stage_a's rows."""
    n = len(plans)
    if n == 0 or len(tables) != n or (prev_ids is not None and len(prev_ids) != n) or \
            (outs is not None and len(outs) != n):
        raise ValueError("stage_a_layers_e4m3: plans, tables, prev_ids and outs must have one entry per layer")
    B, T = ids.shape
    p0 = plans[0]
    if outs is None:
        outs = [(torch.empty(B * T, p.d_mem, dtype=torch.uint8, device=ids.device),
                 torch.empty(B * T, dtype=torch.float32, device=ids.device)) for p in plans]
    arr = lambda vals: (ctypes.c_void_p * n)(*vals)  # noqa: E731
    h = arr([p._h.value for p in plans])
    tab = arr([_dev_or_pinned(t, "table", _TABLE_DTYPES[p.table_dtype][1]) for p, t in zip(plans, tables)])
    prev = 0 if prev_ids is None else arr(
        [0 if x is None else _dev(x, "prev_ids", torch.int32, (B, p.N - 1)) for p, x in zip(plans, prev_ids)])
    q = arr([_dev(o[0], "e8_out", torch.uint8, (B * T, p.d_mem)) for p, o in zip(plans, outs)])
    sc = arr([_dev(o[1], "e_scale_out", torch.float32, (B * T,)) for p, o in zip(plans, outs)])
    _lib.check(p0._lib.engram_stage_a_layers_e4m3(n, h, _dev(ids, "ids", torch.int32), B, T,
                                                  _dev(proj, "proj", torch.int32), proj.numel(), prev, tab, q, sc,
                                                  _stream()), "engram_stage_a_layers_e4m3")
    return list(outs)


def _copy_streams(dev):
    """The host-to-device and device-to-host copy streams of a device, shared by
    every EngramLayer on it so that their transfers cross the link in order."""
    key = torch.device(dev).index
    if key not in _COPY_STREAMS:
        _COPY_STREAMS[key] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    return _COPY_STREAMS[key]


class EngramLayer:
    """A plan, its weights, the projection map and a reusable workspace.

    Calling it runs the whole layer.  With H on the device it is one
    engram_forward.  With H (and ids) in host memory the layer is pipelined
    in ``chunks`` pieces over three streams: the copy of piece i+1 to the
    device, the layer on piece i and the copy of piece i-1 back to the host
    overlap (use pinned host tensors, or the copies serialise).  A piece's
    token ids cross first, and its Stage A (engram_stage_a: Steps 1-4, which
    need the ids only) runs while its H still crosses the link; its Stage B
    (engram_stage_b) follows once H has arrived.  Pieces split
    the batch when B >= chunks (sequences are independent), else the
    positions of a single-sequence batch with a streaming state carried from
    piece to piece; both give the bits of one whole-batch call.  A state
    given with a batch split continues each piece's own sequences.

    The copy streams are shared by all layers on a device.  A call's input
    copies wait for the work already queued on the current stream, or, given
    ``after`` (an event recorded on the current stream), only for that event
    and the same layer's previous call (whose device buffers they reuse): so
    independent layers called one after another with the same ``after``
    overlap, the next layer's inputs crossing while this one computes.  With
    ``join=False`` the current stream does not wait for this call's copy back
    to the host; ``join()`` makes it wait (call it before reading H on the
    host, and before the end of a CUDA-graph capture)."""

    def __init__(self, plan: EngramPlan, weights: EngramWeights, proj: torch.Tensor, chunks: int = 4):
        self.plan, self.weights, self.proj = plan, weights, proj
        self.chunks = max(1, int(chunks))
        self._ws = None
        self._dev_buf = None
        self._e_buf = None
        # (event, recorded during a graph capture): the previous call is done with the device
        # buffers; its copy back to the host completed.  An event is waited on only in the mode
        # it was recorded in: a capture may not wait on eager work (which a capture follows
        # anyway, from a synchronised device), nor eager work on a captured event.
        self._free = None
        self._last_out = None

    def workspace(self, ntok: int, device) -> torch.Tensor:
        need = self.plan.workspace_bytes(ntok)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(max(1, need), dtype=torch.uint8, device=device)
        return self._ws

    def _rows_buffer(self, ntok: int, dev) -> torch.Tensor:
        """Gathered rows e [ntok, d_mem] for Stage A of one piece (reused)."""
        p = self.plan
        if self._e_buf is None or self._e_buf.shape[0] < ntok:
            self._e_buf = torch.empty(max(1, ntok), p.d_mem, dtype=p.act_torch_dtype, device=dev)
        return self._e_buf[:ntok]

    def _buffers(self, ids: torch.Tensor, H: torch.Tensor, dev):
        key = (tuple(ids.shape), tuple(H.shape), H.dtype)
        if self._dev_buf is None or self._dev_buf[0] != key:
            self._dev_buf = (key, torch.empty(ids.shape, dtype=ids.dtype, device=dev),
                             torch.empty(H.shape, dtype=H.dtype, device=dev))
        return self._dev_buf[1], self._dev_buf[2]

    def join(self) -> None:
        """Make the current stream wait for the last call's copy back to the host."""
        if self._last_out is not None and self._last_out[1] == torch.cuda.is_current_stream_capturing():
            torch.cuda.current_stream(self.proj.device).wait_event(self._last_out[0])

    def __call__(self, ids: torch.Tensor, H: torch.Tensor, state: Optional[EngramState] = None,
                 join: bool = True, after: Optional[torch.cuda.Event] = None) -> torch.Tensor:
        dev = self.proj.device
        if H.is_cuda:
            ids_d = ids if ids.is_cuda else ids.to(dev, non_blocking=True)
            self.plan.forward(ids_d, self.proj, self.weights, H, state, self.workspace(ids.numel(), dev))
            return H
        B, T = ids.shape
        if B >= self.chunks and self.chunks > 1:
            cuts = [(B * i // self.chunks, B * (i + 1) // self.chunks) for i in range(self.chunks)]
            along_b = True
        elif B == 1 and state is None and self.chunks > 1 and T >= self.chunks:
            cuts = [(T * i // self.chunks, T * (i + 1) // self.chunks) for i in range(self.chunks)]
            along_b = False
        else:
            cuts = [(0, B)]
            along_b = True
        ids_h = ids if not ids.is_cuda else ids.cpu()
        ids_d, H_d = self._buffers(ids_h, H, dev)
        s_in, s_out = _copy_streams(dev)
        main = torch.cuda.current_stream(dev)
        if after is None:
            after = torch.cuda.Event()
            after.record(main)                    # work the caller queued before this call comes first
        s_in.wait_event(after)
        capturing = torch.cuda.is_current_stream_capturing()
        if self._free is not None and self._free[1] == capturing:
            s_in.wait_event(self._free[0])        # this layer's device buffers are free again
        st = None if along_b else EngramState.zeros(self.plan, 1, dev)
        ws = self.workspace(max(hi - lo for lo, hi in cuts) * (T if along_b else 1), dev)
        last_out = None
        for lo, hi in cuts:
            sl = (slice(lo, hi), slice(None)) if along_b else (slice(None), slice(lo, hi))
            i_h, i_d = ids_h[sl], ids_d[sl]
            h_h, h_d = H[sl], H_d[sl]
            with torch.cuda.stream(s_in):
                i_d.copy_(i_h, non_blocking=True)
                ids_ready = torch.cuda.Event()
                ids_ready.record(s_in)
                h_d.copy_(h_h, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            main.wait_event(ids_ready)
            i_c = i_d if along_b else i_d.contiguous()
            pst = (None if state is None else state.rows(lo, hi)) if along_b else st
            # Stage A needs the ids only: it runs while this piece's H still crosses the link
            e = self.plan.stage_a(i_c, self.proj, self.weights.table, self.weights.scales,
                                  prev_ids=None if pst is None else pst.prev_ids,
                                  out=self._rows_buffer(i_c.numel(), dev))
            main.wait_event(ready)
            h_c = h_d if along_b else h_d.contiguous()
            self.plan.stage_b(e, self.weights, h_c, pst, ids=i_c, proj=self.proj, workspace=ws)
            done = torch.cuda.Event()
            done.record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                h_h.copy_(h_c, non_blocking=True)
                last_out = torch.cuda.Event()
                last_out.record(s_out)
        self._free = (last_out, capturing)        # the last reader of the device buffers
        self._last_out = (last_out, capturing)
        if join:
            main.wait_event(last_out)             # the host copy is complete when main's work is
        return H
