"""ctypes wrapper of the plain-C oracle (test infrastructure only).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark use this
module. It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_u8p = C.POINTER(C.c_uint8)
_u16p = C.POINTER(C.c_uint16)
_i32p = C.POINTER(C.c_int32)
_f32p = C.POINTER(C.c_float)
_f64p = C.POINTER(C.c_double)
_u32p = C.POINTER(C.c_uint32)
_i64p = C.POINTER(C.c_int64)


def _p(a: Optional[np.ndarray], t):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(t)


class Oracle:
    """One loaded build of the oracle library."""

    def __init__(self, path: Optional[str] = None, mutant: int = 0, openmp: bool = True):
        self.path = path or _build.build(mutant=mutant, openmp=openmp)
        self.lib = C.CDLL(self.path)
        L = self.lib
        L.coli_oracle_e2m1.restype = C.c_double
        L.coli_oracle_e2m1.argtypes = [C.c_int]
        L.coli_oracle_e8m0.restype = C.c_double
        L.coli_oracle_e8m0.argtypes = [C.c_int]
        L.coli_oracle_mxfp4.restype = C.c_double
        L.coli_oracle_mxfp4.argtypes = [_u8p, _u8p, C.c_int64, C.c_int64, C.c_int64]
        L.coli_oracle_bf16.restype = C.c_double
        L.coli_oracle_bf16.argtypes = [C.c_uint16]
        L.coli_oracle_round_bf16.restype = C.c_uint16
        L.coli_oracle_round_bf16.argtypes = [C.c_double]
        L.coli_oracle_router_logits.argtypes = [_u16p, C.c_int32, C.c_int32, _f32p, C.c_int32, _f64p]
        L.coli_oracle_sigmoid.argtypes = [_f64p, C.c_int64, _f32p]
        L.coli_oracle_route.argtypes = [_f32p, _f32p, C.c_int32, C.c_int32, C.c_int32, _i32p, _f32p]
        L.coli_oracle_permute.argtypes = [_i32p, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                          _i32p, _i32p, _i32p, _i32p]
        L.coli_oracle_expert_row.argtypes = [_u16p, C.c_int32, C.c_int32, _u8p, _u8p, _u8p, _u8p, _f64p, _f64p]
        L.coli_oracle_tokens_output.argtypes = [_u16p, C.c_int32, C.c_int32, C.c_int32, _i32p, _f32p, C.c_int32,
                                                _u8p, _u8p, _u8p, _u8p, _u8p, _u8p, _u8p, _u8p,
                                                _i32p, C.c_int32, _u16p, _f64p]
        L.coli_oracle_moe_forward.argtypes = [_u16p, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                              _f32p, _f32p, C.c_int32,
                                              _u8p, _u8p, _u8p, _u8p, _u8p, _u8p, _u8p, _u8p,
                                              _f32p, _i32p, _f32p, _i32p, _i32p, _i32p, _i32p, _u16p, _f64p]
        L.coli_oracle_bank_plan.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int32, _i32p,
                                            _i32p, _i32p, _u32p, _i32p, _i64p, _i32p, _i32p, _i32p]
        L.coli_oracle_e4m3.restype = C.c_double
        L.coli_oracle_e4m3.argtypes = [C.c_int]
        L.coli_oracle_fp8_linear.argtypes = [_u16p, C.c_int32, C.c_int32, _u8p, _f32p, C.c_int32, _u16p, _f64p]
        L.coli_oracle_nvfp4.restype = C.c_double
        L.coli_oracle_nvfp4.argtypes = [_u8p, _u8p, C.c_float, C.c_int64, C.c_int64, C.c_int64]
        L.coli_oracle_tokens_output_nv.argtypes = [_u16p, C.c_int32, C.c_int32, C.c_int32, _i32p, _f32p, C.c_int32,
                                                   _u8p, _u8p, _f32p, _u8p, _u8p, _f32p,
                                                   _u8p, _u8p, C.c_float, _u8p, _u8p, C.c_float,
                                                   _i32p, C.c_int32, _u16p, _f64p]
        L.coli_oracle_threads.restype = C.c_int32
        L.coli_oracle_mutant.restype = C.c_int32

    # ---- formats
    def e2m1(self, code: int) -> float:
        return self.lib.coli_oracle_e2m1(code)

    def e8m0(self, s: int) -> float:
        return self.lib.coli_oracle_e8m0(s)

    def mxfp4(self, codes: np.ndarray, scales: np.ndarray, K: int, row: int, k: int) -> float:
        return self.lib.coli_oracle_mxfp4(_p(codes, _u8p), _p(scales, _u8p), K, row, k)

    def e4m3(self, code: int) -> float:
        return self.lib.coli_oracle_e4m3(code)

    def fp8_linear(self, x: np.ndarray, w: np.ndarray, w_scale: np.ndarray):
        """out bf16 bits [T, N] and fp64 sums of x [T, K] (bf16 bits) times the E4M3 block-scaled w [N, K]."""
        x = np.ascontiguousarray(x, np.uint16)
        w = np.ascontiguousarray(w, np.uint8)
        sc = np.ascontiguousarray(w_scale, np.float32)
        T, K = x.shape
        N = w.shape[0]
        out = np.zeros((T, N), np.uint16)
        out64 = np.zeros((T, N), np.float64)
        self.lib.coli_oracle_fp8_linear(_p(x, _u16p), T, K, _p(w, _u8p), _p(sc, _f32p), N, _p(out, _u16p),
                                        _p(out64, _f64p))
        return out, out64

    def bf16(self, bits: int) -> float:
        return self.lib.coli_oracle_bf16(bits)

    def round_bf16(self, v: float) -> int:
        return self.lib.coli_oracle_round_bf16(v)

    def threads(self) -> int:
        return self.lib.coli_oracle_threads()

    def mutant(self) -> int:
        return self.lib.coli_oracle_mutant()

    # ---- router
    def router_logits(self, x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
        T, H = x.shape
        E = router_w.shape[0]
        out = np.zeros((T, E), np.float64)
        self.lib.coli_oracle_router_logits(_p(x, _u16p), T, H, _p(router_w, _f32p), E, _p(out, _f64p))
        return out

    def sigmoid(self, logits: np.ndarray) -> np.ndarray:
        logits = np.ascontiguousarray(logits, np.float64)
        s = np.zeros(logits.shape, np.float32)
        self.lib.coli_oracle_sigmoid(_p(logits, _f64p), logits.size, _p(s, _f32p))
        return s

    def scores(self, x: np.ndarray, router_w: np.ndarray) -> np.ndarray:
        return self.sigmoid(self.router_logits(x, router_w))

    def route(self, s: np.ndarray, router_b: Optional[np.ndarray], top_k: int):
        s = np.ascontiguousarray(s, np.float32)
        T, E = s.shape
        idx = np.zeros((T, top_k), np.int32)
        w = np.zeros((T, top_k), np.float32)
        b = None if router_b is None else np.ascontiguousarray(router_b, np.float32)
        self.lib.coli_oracle_route(_p(s, _f32p), _p(b, _f32p), T, E, top_k, _p(idx, _i32p), _p(w, _f32p))
        return idx, w

    # ---- permute
    def permute(self, idx: np.ndarray, E: int, with_shared: bool = True):
        idx = np.ascontiguousarray(idx, np.int32)
        T, k = idx.shape
        cnt = np.zeros(E + 1, np.int32)
        off = np.zeros(E + 2, np.int32)
        src = np.full(T * k + T, -1, np.int32)
        inv = np.full((T, k), -1, np.int32)
        self.lib.coli_oracle_permute(_p(idx, _i32p), T, E, k, int(with_shared), _p(cnt, _i32p), _p(off, _i32p),
                                     _p(src, _i32p), _p(inv, _i32p))
        rows = int(off[E + 1])
        return cnt, off, src[:rows].copy(), inv

    # ---- FFN
    def expert_row(self, x_row: np.ndarray, gu_codes, gu_scales, d_codes, d_scales):
        H = x_row.shape[0]
        I = gu_codes.shape[0] // 2
        y = np.zeros(H, np.float64)
        h = np.zeros(I, np.float64)
        self.lib.coli_oracle_expert_row(_p(np.ascontiguousarray(x_row), _u16p), H, I,
                                        _p(gu_codes, _u8p), _p(gu_scales, _u8p),
                                        _p(d_codes, _u8p), _p(d_scales, _u8p), _p(y, _f64p), _p(h, _f64p))
        return y, h

    def tokens_output(self, x: np.ndarray, idx: np.ndarray, w: np.ndarray, experts, shared,
                      tokens: Sequence[int]):
        """Output rows (bf16 bits, fp64 sums) for the listed tokens given routing idx/w."""
        T, H = x.shape
        k = idx.shape[1]
        I = experts.gate_up_codes.shape[1] // 2
        I_s = shared.gate_up_codes.shape[1] // 2 if shared is not None else 0
        tok = np.ascontiguousarray(np.asarray(tokens, np.int32))
        out = np.zeros((len(tok), H), np.uint16)
        out64 = np.zeros((len(tok), H), np.float64)
        sh = [None] * 4 if shared is None else [shared.gate_up_codes, shared.gate_up_scales,
                                                 shared.down_codes, shared.down_scales]
        self.lib.coli_oracle_tokens_output(
            _p(x, _u16p), H, I, I_s, _p(np.ascontiguousarray(idx, np.int32), _i32p),
            _p(np.ascontiguousarray(w, np.float32), _f32p), k,
            _p(experts.gate_up_codes, _u8p), _p(experts.gate_up_scales, _u8p),
            _p(experts.down_codes, _u8p), _p(experts.down_scales, _u8p),
            *[_p(a, _u8p) for a in sh], _p(tok, _i32p), len(tok), _p(out, _u16p), _p(out64, _f64p))
        return out, out64

    def nvfp4(self, codes: np.ndarray, scales: np.ndarray, glob: float, K: int, row: int, k: int) -> float:
        return self.lib.coli_oracle_nvfp4(_p(codes, _u8p), _p(scales, _u8p), glob, K, row, k)

    def tokens_output_nv(self, x: np.ndarray, idx: np.ndarray, w: np.ndarray, experts, shared,
                         tokens: Sequence[int]):
        """tokens_output with NVFP4 experts (synthetic.NVFP4Experts)."""
        T, H = x.shape
        k = idx.shape[1]
        I = experts.gate_up_codes.shape[1] // 2
        I_s = shared.gate_up_codes.shape[1] // 2 if shared is not None else 0
        tok = np.ascontiguousarray(np.asarray(tokens, np.int32))
        out = np.zeros((len(tok), H), np.uint16)
        out64 = np.zeros((len(tok), H), np.float64)
        if shared is None:
            sh = [None, None, 0.0, None, None, 0.0]
        else:
            sh = [_p(shared.gate_up_codes, _u8p), _p(shared.gate_up_scales, _u8p), float(shared.gate_up_global[0]),
                  _p(shared.down_codes, _u8p), _p(shared.down_scales, _u8p), float(shared.down_global[0])]
        self.lib.coli_oracle_tokens_output_nv(
            _p(x, _u16p), H, I, I_s, _p(np.ascontiguousarray(idx, np.int32), _i32p),
            _p(np.ascontiguousarray(w, np.float32), _f32p), k,
            _p(experts.gate_up_codes, _u8p), _p(experts.gate_up_scales, _u8p),
            _p(np.ascontiguousarray(experts.gate_up_global, np.float32), _f32p),
            _p(experts.down_codes, _u8p), _p(experts.down_scales, _u8p),
            _p(np.ascontiguousarray(experts.down_global, np.float32), _f32p),
            *sh, _p(tok, _i32p), len(tok), _p(out, _u16p), _p(out64, _f64p))
        return out, out64

    def moe_forward(self, x: np.ndarray, router_w: np.ndarray, router_b: Optional[np.ndarray], top_k: int,
                    experts, shared):
        """The whole layer through the permuted path; returns a dict of every intermediate."""
        T, H = x.shape
        E = router_w.shape[0]
        I = experts.gate_up_codes.shape[1] // 2
        I_s = shared.gate_up_codes.shape[1] // 2 if shared is not None else 0
        s = np.zeros((T, E), np.float32)
        idx = np.zeros((T, top_k), np.int32)
        w = np.zeros((T, top_k), np.float32)
        cnt = np.zeros(E + 1, np.int32)
        off = np.zeros(E + 2, np.int32)
        src = np.full(T * top_k + T, -1, np.int32)
        inv = np.full((T, top_k), -1, np.int32)
        out = np.zeros((T, H), np.uint16)
        out64 = np.zeros((T, H), np.float64)
        b = None if router_b is None else np.ascontiguousarray(router_b, np.float32)
        sh = [None] * 4 if shared is None else [shared.gate_up_codes, shared.gate_up_scales,
                                                 shared.down_codes, shared.down_scales]
        self.lib.coli_oracle_moe_forward(
            _p(x, _u16p), T, H, E, I, I_s, _p(router_w, _f32p), _p(b, _f32p), top_k,
            _p(experts.gate_up_codes, _u8p), _p(experts.gate_up_scales, _u8p),
            _p(experts.down_codes, _u8p), _p(experts.down_scales, _u8p),
            *[_p(a, _u8p) for a in sh],
            _p(s, _f32p), _p(idx, _i32p), _p(w, _f32p), _p(cnt, _i32p), _p(off, _i32p),
            _p(src, _i32p), _p(inv, _i32p), _p(out, _u16p), _p(out64, _f64p))
        rows = int(off[E + 1])
        return dict(s=s, idx=idx, w=w, cnt=cnt, off=off, src_token=src[:rows].copy(), inv_row=inv,
                    out=out, out_f64=out64)


class BankState:
    """Host copy of an expert residency bank's state (the oracle's bank plan updates it)."""

    def __init__(self, E: int, S: int):
        self.E, self.S = E, S
        self.slot_of = np.full(E, -1, np.int32)
        self.expert_in = np.full(S, -1, np.int32)
        self.usage = np.zeros(E, np.uint32)
        self.last_use = np.zeros(S, np.int32)
        self.stats = np.zeros(3, np.int64)

    def copy(self) -> "BankState":
        c = BankState(self.E, self.S)
        for k in ("slot_of", "expert_in", "usage", "last_use", "stats"):
            setattr(c, k, getattr(self, k).copy())
        return c


def bank_plan(o: Oracle, state: BankState, cnt: np.ndarray, T: int, top_k: int):
    """One forward's effect on the bank (state updated in place); returns per-expert
    (round_of, slot_for, copied)."""
    E, S = state.E, state.S
    cnt = np.ascontiguousarray(cnt[:E], np.int32)
    rnd = np.zeros(E, np.int32)
    slot = np.zeros(E, np.int32)
    cop = np.zeros(E, np.int32)
    o.lib.coli_oracle_bank_plan(E, S, T, top_k, _p(cnt, _i32p), _p(state.slot_of, _i32p),
                                _p(state.expert_in, _i32p), _p(state.usage, _u32p), _p(state.last_use, _i32p),
                                _p(state.stats, _i64p), _p(rnd, _i32p), _p(slot, _i32p), _p(cop, _i32p))
    return rnd, slot, cop


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
