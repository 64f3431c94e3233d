"""Thin Python binding of libdd (include/dd.h, include/dd_synth.h).

Argument marshalling only: every function checks the tensors it is given
(device, dtype, size, contiguity), passes their addresses and the current CUDA
stream to the C ABI, and raises ``DDError`` on a non-OK status.  All compute
runs in the library's CUDA kernels; there is no fallback -- importing this
module without a built ``libdd.so`` raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libdd.so")

DD_OK, DD_ERR_INVALID_ARG, DD_ERR_CUDA, DD_ERR_CAPACITY, DD_ERR_TIMEOUT, DD_ERR_DEVICE_CHECK = range(6)
GATHER_ZEROCOPY, GATHER_MEMCPY, GATHER_KERNEL, GATHER_AUTO = 0, 1, 2, 3
TRACE_SLOTS = 256          # per-SM slots of a step's timing words (DD_TRACE_SLOTS)
LM_MEAN, LM_MINMAX = 0, 1

EXPORTED = (
    "dd_create", "dd_destroy", "dd_build_landmarks", "dd_score_landmarks", "dd_select_topk",
    "dd_resolve_union", "dd_gather_kv", "dd_sparse_attn_decode", "dd_step", "dd_get_status",
    "dd_launch_count", "dd_status_str", "dd_last_cuda_error", "dd_synth_kv", "dd_synth_queries", "dd_sparse_attn_decode_noalloc",
    "dd_build_landmarks_minmax", "dd_score_landmarks_minmax", "dd_update_residency",
    "dd_prefetch_kv", "dd_select_topk_mass", "dd_selftest_bounded_wait", "dd_step_folds_scoring",
)


class DDError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == DD_ERR_CUDA:
            detail = " [" + _lib.dd_last_cuda_error().decode() + "]"
        super().__init__(f"{what}: {status_str(status)} ({status}){detail}")


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "Hq", "Hkv", "d", "L", "cs", "k", "n_q")]


_vp = ctypes.c_void_p


class StepArgs(ctypes.Structure):
    _fields_ = [
        ("layer", ctypes.c_int32), ("q", _vp), ("lm", _vp), ("Kh", _vp), ("Vh", _vp),
        ("resident_slot", _vp), ("Khot", _vp), ("Vhot", _vp), ("Kst", _vp * 2), ("Vst", _vp * 2),
        ("mode", ctypes.c_int), ("softmax_scale", ctypes.c_float), ("out", _vp),
        ("scores", _vp), ("sel", _vp), ("union_idx", _vp), ("union_slot", _vp), ("union_cnt", _vp),
        ("miss_list", _vp), ("miss_count", _vp), ("attn_slot", _vp), ("union_qmask", _vp),
        ("stage_events", _vp * 6),
        ("lm_kind", ctypes.c_int),
        ("K_tail", _vp),
        ("V_tail", _vp),
        ("mass_gamma", ctypes.c_float),
        ("mass_k_min", ctypes.c_int32),
        ("sel_cnt", _vp),
        ("trace", _vp),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libdd.so is not built ({LIB_PATH}); run sparse_kv_offload_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sig = {
        "dd_create": (i32, [ctypes.POINTER(Dims), i64, i64, ctypes.POINTER(_vp)]),
        "dd_destroy": (i32, [_vp]),
        "dd_build_landmarks": (i32, [_vp, _vp, _vp, _vp]),
        "dd_score_landmarks": (i32, [_vp, _vp, _vp, _vp, _vp]),
        "dd_build_landmarks_minmax": (i32, [_vp, _vp, _vp, _vp]),
        "dd_score_landmarks_minmax": (i32, [_vp, _vp, _vp, _vp, _vp]),
        "dd_select_topk": (i32, [_vp, _vp, _vp, _vp]),
        "dd_resolve_union": (i32, [_vp] * 11),
        "dd_gather_kv": (i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp]),
        "dd_sparse_attn_decode": (i32, [_vp] * 12 + [f32, _vp, _vp]),
        "dd_step": (i32, [_vp, ctypes.POINTER(StepArgs), _vp]),
        "dd_update_residency": (i32, [_vp, i32, i32, i32] + [_vp] * 13),
        "dd_selftest_bounded_wait": (i32, [_vp, i32, _vp]),
        "dd_select_topk_mass": (i32, [_vp, _vp, _vp, _vp, f32, i32, f32, _vp]),
        "dd_prefetch_kv": (i32, [_vp, _vp, i32, i32, i32, _vp, _vp, _vp, _vp, _vp, _vp, i32, _vp]),
        "dd_get_status": (i32, [_vp, ctypes.POINTER(i32)]),
        "dd_launch_count": (i64, [_vp]),
        "dd_step_folds_scoring": (i32, [ctypes.POINTER(Dims), i32, ctypes.c_int, f32]),
        "dd_status_str": (ctypes.c_char_p, [i32]),
        "dd_last_cuda_error": (ctypes.c_char_p, []),
        "dd_synth_kv": (i32, [ctypes.POINTER(Dims), ctypes.c_uint64, i32, _vp, _vp, _vp, i64, _vp, _vp]),
        "dd_synth_queries": (i32, [ctypes.POINTER(Dims), ctypes.c_uint64, i32, ctypes.POINTER(f32), _vp, _vp]),
        "dd_sparse_attn_decode_noalloc": (i32, [ctypes.POINTER(Dims), i64, i64] + [_vp] * 9 + [f32, _vp, _vp, _vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def status_str(s: int) -> str:
    return _lib.dd_status_str(int(s)).decode()


def _chk(status: int, what: str):
    if status != DD_OK:
        raise DDError(status, what)


def _stream(stream) -> int:
    # the current stream's raw handle without building a torch.cuda.Stream
    # object (a tenth of the host time of torch.cuda.current_stream())
    if stream is not None:
        return stream.cuda_stream
    return torch._C._cuda_getCurrentRawStream(torch._C._cuda_getDevice())


def _ptr(t, dtype=None, numel=None, device=True, name="tensor", allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not device and (t.is_cuda or not t.is_pinned()):
        raise ValueError(f"{name} must be a pinned host tensor")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


@dataclass(frozen=True)
class Shape:
    B: int
    Hq: int
    Hkv: int
    d: int
    L: int
    cs: int
    k: int
    n_q: int

    @property
    def C(self):
        return self.L // self.cs

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def umax(self):
        return min(self.C, self.n_q * self.k)

    def dims(self) -> Dims:
        return Dims(self.B, self.Hq, self.Hkv, self.d, self.L, self.cs, self.k, self.n_q)


def step_folds_scoring(shape: "Shape", sm_count: int, lm_kind: int = 0, mass_gamma: float = 0.0) -> int:
    """Ring depth of the selection kernel that scores its own unit inside dd_step
    (0: the step runs the scoring kernel first); host only."""
    d = shape.dims()
    return int(_lib.dd_step_folds_scoring(ctypes.byref(d), int(sm_count), int(lm_kind), float(mass_gamma)))


class Context:
    """One libdd context (workspace, status word, events, copy stream) on the current device."""

    def __init__(self, shape: Shape, max_misses: int, hot_slots: int = 0):
        self.shape = shape
        self.max_misses = int(max_misses)
        self.hot_slots = int(hot_slots)
        self._dims = shape.dims()
        h = _vp()
        _chk(_lib.dd_create(ctypes.byref(self._dims), self.max_misses, self.hot_slots, ctypes.byref(h)), "dd_create")
        self._h = h

    def close(self):
        if self._h:
            _lib.dd_destroy(self._h)
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

    # ------------------------------------------------------------------ stages
    def build_landmarks(self, K, lm, stream=None):
        s = self.shape
        n = s.B * s.Hkv * s.L * s.d
        kp = _ptr(K, torch.bfloat16, n, device=K.is_cuda, name="K")
        _chk(_lib.dd_build_landmarks(self._h, kp, _ptr(lm, torch.bfloat16, s.B * s.Hkv * s.C * s.d, name="lm"),
                                     _stream(stream)), "dd_build_landmarks")

    def score_landmarks(self, q, lm, scores, stream=None):
        s = self.shape
        _chk(_lib.dd_score_landmarks(
            self._h, _ptr(q, torch.bfloat16, s.B * s.n_q * s.Hq * s.d, name="q"),
            _ptr(lm, torch.bfloat16, s.B * s.Hkv * s.C * s.d, name="lm"),
            _ptr(scores, torch.float32, s.B * s.n_q * s.Hkv * s.C, name="scores"), _stream(stream)),
            "dd_score_landmarks")

    def build_landmarks_minmax(self, K, lm2, stream=None):
        s = self.shape
        n = s.B * s.Hkv * s.L * s.d
        kp = _ptr(K, torch.bfloat16, n, device=K.is_cuda, name="K")
        _chk(_lib.dd_build_landmarks_minmax(
            self._h, kp, _ptr(lm2, torch.bfloat16, s.B * s.Hkv * s.C * 2 * s.d, name="lm2"), _stream(stream)),
            "dd_build_landmarks_minmax")

    def score_landmarks_minmax(self, q, lm2, scores, stream=None):
        s = self.shape
        _chk(_lib.dd_score_landmarks_minmax(
            self._h, _ptr(q, torch.bfloat16, s.B * s.n_q * s.Hq * s.d, name="q"),
            _ptr(lm2, torch.bfloat16, s.B * s.Hkv * s.C * 2 * s.d, name="lm2"),
            _ptr(scores, torch.float32, s.B * s.n_q * s.Hkv * s.C, name="scores"), _stream(stream)),
            "dd_score_landmarks_minmax")

    def select_topk(self, scores, sel, stream=None):
        s = self.shape
        _chk(_lib.dd_select_topk(self._h, _ptr(scores, torch.float32, s.B * s.n_q * s.Hkv * s.C, name="scores"),
                                 _ptr(sel, torch.int32, s.B * s.n_q * s.Hkv * s.k, name="sel"), _stream(stream)),
             "dd_select_topk")

    def resolve_union(self, sel, resident_slot, union_idx, union_slot, union_qmask, union_cnt, miss_list,
                      miss_count, attn_slot=None, stream=None):
        s = self.shape
        nu = s.B * s.Hkv * s.umax
        _chk(_lib.dd_resolve_union(
            self._h, _ptr(sel, torch.int32, s.B * s.n_q * s.Hkv * s.k, name="sel"),
            _ptr(resident_slot, torch.int32, s.B * s.Hkv * s.C, name="resident_slot"),
            _ptr(union_idx, torch.int32, nu, name="union_idx"), _ptr(union_slot, torch.int32, nu, name="union_slot"),
            _ptr(union_qmask, torch.uint8, nu, name="union_qmask"),
            _ptr(union_cnt, torch.int32, s.B * s.Hkv, name="union_cnt"),
            _ptr(miss_list, torch.int32, max(1, self.max_misses), name="miss_list"),
            _ptr(miss_count, torch.int32, 1, name="miss_count"),
            _ptr(attn_slot, torch.int32, s.B * s.n_q * s.Hkv * s.k, name="attn_slot", allow_none=True),
            _stream(stream)), "dd_resolve_union")

    def gather_kv(self, Kh, Vh, miss_list, miss_count, Kst, Vst, mode=GATHER_ZEROCOPY, stream=None):
        s = self.shape
        n = s.B * s.Hkv * s.L * s.d
        ns = self.max_misses * s.cs * s.d
        _chk(_lib.dd_gather_kv(
            self._h, _ptr(Kh, torch.bfloat16, n, device=False, name="Kh"),
            _ptr(Vh, torch.bfloat16, n, device=False, name="Vh"),
            _ptr(miss_list, torch.int32, 1, name="miss_list"), _ptr(miss_count, torch.int32, 1, name="miss_count"),
            _ptr(Kst, torch.bfloat16, ns, name="Kst"), _ptr(Vst, torch.bfloat16, ns, name="Vst"), int(mode),
            _stream(stream)), "dd_gather_kv")

    def sparse_attn_decode(self, q, Khot, Vhot, Kst, Vst, union_slot, union_qmask, union_cnt, miss_count, out,
                           softmax_scale=0.0, stream=None, K_tail=None, V_tail=None):
        s = self.shape
        nh = self.hot_slots * s.cs * s.d
        ns = self.max_misses * s.cs * s.d
        nu = s.B * s.Hkv * s.umax
        nt = s.B * s.n_q * s.Hkv * s.d
        _chk(_lib.dd_sparse_attn_decode(
            self._h, _ptr(q, torch.bfloat16, s.B * s.n_q * s.Hq * s.d, name="q"),
            _ptr(Khot, torch.bfloat16, nh, name="Khot", allow_none=True),
            _ptr(Vhot, torch.bfloat16, nh, name="Vhot", allow_none=True),
            _ptr(Kst, torch.bfloat16, ns, name="Kst", allow_none=True),
            _ptr(Vst, torch.bfloat16, ns, name="Vst", allow_none=True),
            _ptr(K_tail, torch.bfloat16, nt, name="K_tail", allow_none=True),
            _ptr(V_tail, torch.bfloat16, nt, name="V_tail", allow_none=True),
            _ptr(union_slot, torch.int32, nu, name="union_slot"), _ptr(union_qmask, torch.uint8, nu, name="union_qmask"),
            _ptr(union_cnt, torch.int32, s.B * s.Hkv, name="union_cnt"),
            _ptr(miss_count, torch.int32, 1, name="miss_count"), float(softmax_scale),
            _ptr(out, torch.float32, s.B * s.n_q * s.Hq * s.d, name="out"), _stream(stream)),
            "dd_sparse_attn_decode")

    def selftest_bounded_wait(self, kind, stream=None):
        """Run a bounded device wait that nothing signals (see dd.h); the status
        word then holds DD_ERR_TIMEOUT."""
        _chk(_lib.dd_selftest_bounded_wait(self._h, int(kind), _stream(stream)), "dd_selftest_bounded_wait")

    def select_topk_mass(self, scores, sel, gamma, k_min=1, sel_cnt=None, softmax_scale=0.0, stream=None):
        """Coverage-budget top-k (see dd.h): rows padded with -1, lengths in sel_cnt."""
        s = self.shape
        rows = s.B * s.n_q * s.Hkv
        _chk(_lib.dd_select_topk_mass(
            self._h, _ptr(scores, torch.float32, rows * s.C, name="scores"),
            _ptr(sel, torch.int32, rows * s.k, name="sel"),
            _ptr(sel_cnt, torch.int32, rows, name="sel_cnt", allow_none=True), float(gamma), int(k_min),
            float(softmax_scale), _stream(stream)), "dd_select_topk_mass")

    def prefetch_kv(self, sel, n_pred, Kh, Vh, Kpf, Vpf, pf_map, pf_count=None, ctas_per_sm=8, stream=None,
                    sel_rows=None, first_row=0):
        """Predictive prefetch of rows first_row .. first_row+n_pred-1 of ``sel``
        [B, sel_rows, Hkv, k] (sel_rows defaults to n_pred; see dd.h)."""
        s = self.shape
        n = s.B * s.Hkv * s.L * s.d
        ns = self.max_misses * s.cs * s.d
        rows = n_pred if sel_rows is None else sel_rows
        _chk(_lib.dd_prefetch_kv(
            self._h, _ptr(sel, torch.int32, s.B * max(rows, 0) * s.Hkv * s.k, name="sel"), int(rows),
            int(first_row), int(n_pred),
            _ptr(Kh, torch.bfloat16, n, device=False, name="Kh"), _ptr(Vh, torch.bfloat16, n, device=False, name="Vh"),
            _ptr(Kpf, torch.bfloat16, ns, name="Kpf", allow_none=True),
            _ptr(Vpf, torch.bfloat16, ns, name="Vpf", allow_none=True),
            _ptr(pf_map, torch.int32, s.B * s.Hkv * s.C, name="pf_map"),
            _ptr(pf_count, torch.int32, 1, name="pf_count", allow_none=True), int(ctas_per_sm), _stream(stream)),
            "dd_prefetch_kv")

    def update_residency(self, step, cap, slots_per_unit, Kst, Vst, resident_slot, slot_chunk, last_used, Khot,
                         Vhot, admitted=None, union_idx=None, union_slot=None, union_cnt=None, miss_count=None,
                         stream=None):
        """Capped LRU residency update after a step (see dd.h); the union arrays default
        to the context's workspace (the last step that used it)."""
        s = self.shape
        units = s.B * s.Hkv
        nu = units * s.umax
        nh = self.hot_slots * s.cs * s.d
        ns = self.max_misses * s.cs * s.d
        _chk(_lib.dd_update_residency(
            self._h, int(step), int(cap), int(slots_per_unit),
            _ptr(union_idx, torch.int32, nu, name="union_idx", allow_none=True),
            _ptr(union_slot, torch.int32, nu, name="union_slot", allow_none=True),
            _ptr(union_cnt, torch.int32, units, name="union_cnt", allow_none=True),
            _ptr(miss_count, torch.int32, 1, name="miss_count", allow_none=True),
            _ptr(Kst, torch.bfloat16, ns, name="Kst", allow_none=True),
            _ptr(Vst, torch.bfloat16, ns, name="Vst", allow_none=True),
            _ptr(resident_slot, torch.int32, units * s.C, name="resident_slot"),
            _ptr(slot_chunk, torch.int32, units * slots_per_unit, name="slot_chunk"),
            _ptr(last_used, torch.int32, units * slots_per_unit, name="last_used"),
            _ptr(Khot, torch.bfloat16, nh, name="Khot"), _ptr(Vhot, torch.bfloat16, nh, name="Vhot"),
            _ptr(admitted, torch.int32, units, name="admitted", allow_none=True), _stream(stream)),
            "dd_update_residency")

    def step(self, layer, q, lm, Kh, Vh, resident_slot, Khot, Vhot, Kst_pair, Vst_pair, out,
             mode=GATHER_ZEROCOPY, softmax_scale=0.0, intermediates=None, stage_events=None, stream=None,
             lm_kind=LM_MEAN, K_tail=None, V_tail=None, mass_gamma=0.0, mass_k_min=1, sel_cnt=None, trace=None):
        """One layer; ``intermediates`` optionally maps names of dd_step_args' optional
        outputs (scores, sel, union_idx, union_slot, union_qmask, union_cnt, miss_list,
        miss_count, attn_slot) to caller tensors; ``stage_events`` optionally gives six
        torch.cuda.Event objects recorded at the stage boundaries; ``lm_kind`` says
        whether ``lm`` holds mean landmarks or min/max landmarks (twice the size)."""
        s = self.shape
        a = StepArgs()
        a.layer = int(layer)
        a.q = _ptr(q, torch.bfloat16, s.B * s.n_q * s.Hq * s.d, name="q")
        a.lm_kind = int(lm_kind)
        a.mass_gamma = float(mass_gamma)
        a.mass_k_min = int(mass_k_min)
        a.sel_cnt = _ptr(sel_cnt, torch.int32, s.B * s.n_q * s.Hkv, name="sel_cnt", allow_none=True)
        # int64 tensor of 3 * 2 * TRACE_SLOTS (uint64 bits): see dd_step_args.trace
        a.trace = _ptr(trace, torch.int64, 6 * TRACE_SLOTS, name="trace", allow_none=True)
        a.K_tail = _ptr(K_tail, torch.bfloat16, s.B * s.n_q * s.Hkv * s.d, name="K_tail", allow_none=True)
        a.V_tail = _ptr(V_tail, torch.bfloat16, s.B * s.n_q * s.Hkv * s.d, name="V_tail", allow_none=True)
        a.lm = _ptr(lm, torch.bfloat16, s.B * s.Hkv * s.C * s.d * (2 if lm_kind == LM_MINMAX else 1), name="lm")
        n = s.B * s.Hkv * s.L * s.d
        a.Kh = _ptr(Kh, torch.bfloat16, n, device=False, name="Kh")
        a.Vh = _ptr(Vh, torch.bfloat16, n, device=False, name="Vh")
        a.resident_slot = _ptr(resident_slot, torch.int32, s.B * s.Hkv * s.C, name="resident_slot")
        nh = self.hot_slots * s.cs * s.d
        a.Khot = _ptr(Khot, torch.bfloat16, nh, name="Khot", allow_none=True)
        a.Vhot = _ptr(Vhot, torch.bfloat16, nh, name="Vhot", allow_none=True)
        ns = self.max_misses * s.cs * s.d
        for p in range(2):
            a.Kst[p] = _ptr(Kst_pair[p], torch.bfloat16, ns, name="Kst", allow_none=True)
            a.Vst[p] = _ptr(Vst_pair[p], torch.bfloat16, ns, name="Vst", allow_none=True)
        a.mode = int(mode)
        a.softmax_scale = float(softmax_scale)
        a.out = _ptr(out, torch.float32, s.B * s.n_q * s.Hq * s.d, name="out")
        for name, t in (intermediates or {}).items():
            dt = {"scores": torch.float32, "union_qmask": torch.uint8}.get(name, torch.int32)
            setattr(a, name, _ptr(t, dt, 1, name=name))
        for i, ev in enumerate(stage_events or ()):
            if ev is not None:
                a.stage_events[i] = ev.cuda_event
        self._last_args = a
        _chk(_lib.dd_step(self._h, ctypes.byref(a), _stream(stream)), "dd_step")

    def status(self) -> int:
        """Wait for the device, return and clear the device status word."""
        v = ctypes.c_int32(0)
        _chk(_lib.dd_get_status(self._h, ctypes.byref(v)), "dd_get_status")
        return int(v.value)

    def launch_count(self) -> int:
        return int(_lib.dd_launch_count(self._h))


# ---------------------------------------------------------------- allocation-free attention
def sparse_attn_decode_noalloc(shape: Shape, hot_slots, max_misses, q, Khot, Vhot, Kst, Vst, union_slot,
                               union_qmask, union_cnt, miss_count, out, device_status, softmax_scale=0.0,
                               stream=None):
    """dd_sparse_attn_decode without a context, for callers that cannot
    allocate device memory: its split-K partials sit in the library's fixed
    16 MiB device array.  ``device_status`` is a zeroed device int32 tensor that
    receives a device-detected dd_status code.  Calls that overlap on the GPU
    share that array and race; serialise them."""
    s = shape
    dims = s.dims()
    nh = int(hot_slots) * s.cs * s.d
    ns = int(max_misses) * s.cs * s.d
    nu = s.B * s.Hkv * s.umax
    _chk(_lib.dd_sparse_attn_decode_noalloc(
        ctypes.byref(dims), int(hot_slots), int(max_misses),
        _ptr(q, torch.bfloat16, s.B * s.n_q * s.Hq * s.d, name="q"),
        _ptr(Khot, torch.bfloat16, nh, name="Khot", allow_none=True),
        _ptr(Vhot, torch.bfloat16, nh, name="Vhot", allow_none=True),
        _ptr(Kst, torch.bfloat16, ns, name="Kst", allow_none=True),
        _ptr(Vst, torch.bfloat16, ns, name="Vst", allow_none=True),
        _ptr(union_slot, torch.int32, nu, name="union_slot"), _ptr(union_qmask, torch.uint8, nu, name="union_qmask"),
        _ptr(union_cnt, torch.int32, s.B * s.Hkv, name="union_cnt"), _ptr(miss_count, torch.int32, 1, name="miss_count"),
        float(softmax_scale), _ptr(out, torch.float32, s.B * s.n_q * s.Hq * s.d, name="out"),
        _ptr(device_status, torch.int32, 1, name="device_status"), _stream(stream)),
        "dd_sparse_attn_decode_noalloc")


# ---------------------------------------------------------------- generator
def synth_kv(shape: Shape, seed: int, tensor_id: int, dst, bias=None, u_hat=None, chunk_map=None, stream=None):
    dims = shape.dims()
    n_slots = 0 if chunk_map is None else int(chunk_map.numel())
    numel = n_slots * shape.cs * shape.d if chunk_map is not None else shape.B * shape.Hkv * shape.L * shape.d
    dp = _ptr(dst, torch.bfloat16, numel, device=dst.is_cuda, name="dst")
    _chk(_lib.dd_synth_kv(ctypes.byref(dims), int(seed), int(tensor_id),
                          _ptr(bias, torch.float32, shape.B * shape.Hkv * shape.C, name="bias", allow_none=True),
                          _ptr(u_hat, torch.float32, shape.B * shape.Hkv * shape.d, name="u_hat", allow_none=True),
                          _ptr(chunk_map, torch.int32, n_slots, name="chunk_map", allow_none=True), n_slots, dp,
                          _stream(stream)), "dd_synth_kv")


def synth_queries(shape: Shape, seed: int, layer: int, spec_scale, dst, stream=None):
    dims = shape.dims()
    sc = (ctypes.c_float * max(1, shape.n_q))(*[float(x) for x in list(spec_scale)[:shape.n_q]])
    _chk(_lib.dd_synth_queries(ctypes.byref(dims), int(seed), int(layer), sc,
                               _ptr(dst, torch.bfloat16, shape.B * shape.n_q * shape.Hq * shape.d, name="q"),
                               _stream(stream)), "dd_synth_queries")


def default_scale(d: int = 128) -> float:
    return 1.0 / math.sqrt(d)
