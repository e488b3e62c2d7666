"""CPU oracle for the top-k MoE layer forward -- TEST INFRASTRUCTURE.

A plain, slow, single-threaded fp64 definition of the layer (``moe_oracle.cpp``),
wrapped for numpy. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it. It shares no code with the CUDA library
and never imports it; the library never imports this package.

Arrays are numpy: fp32 arrays, or bf16 tensors passed as their uint16 bit
patterns (``dtype="bf16"``). The wrapper only marshals arguments and composes
the C functions in the order the layer defines:

    logits -> top-k -> gates -> capacity/dropping -> expert outputs -> combine

Which page passage each step follows is stated in ``moe_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
LIB_PATH = os.path.join(_HERE, "liboracle.so")

GATING = {"softmax_topk": 0, "softmax_topk_renorm": 1, "topk_softmax": 2, "expert_choice": 3}
ACT = {"gelu": 0, "swiglu": 1}


def build(out_path: str = LIB_PATH, plant: int = 0, force: bool = False) -> str:
    """Compile the oracle with g++ (``plant`` != 0 compiles in a deliberate mistake)."""
    if not force and plant == 0 and os.path.exists(out_path) and \
            os.path.getmtime(out_path) >= os.path.getmtime(_SRC):
        return out_path
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", f"-DORACLE_PLANT={plant}", "-o", out_path, _SRC]
    subprocess.run(cmd, check=True)
    return out_path


class OracleConfig(ctypes.Structure):
    _fields_ = [
        ("n_tokens", ctypes.c_int64), ("d_model", ctypes.c_int64), ("d_ff", ctypes.c_int64),
        ("n_experts", ctypes.c_int64), ("n_shared", ctypes.c_int64), ("d_ff_shared", ctypes.c_int64),
        ("top_k", ctypes.c_int64), ("capacity_factor", ctypes.c_double), ("gating", ctypes.c_int32),
        ("act", ctypes.c_int32), ("has_bias", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("aux_alpha", ctypes.c_double), ("mimic_bf16", ctypes.c_int32), ("passthrough", ctypes.c_int32),
        ("mx_act", ctypes.c_int32),
    ]


class OracleWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_router", "logit_bias", "w1", "w3", "b1", "w2", "b2", "ws1", "ws3", "bs1", "ws2", "bs2")]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, lib_path: Optional[str] = None):
        path = lib_path or build()
        lib = ctypes.CDLL(path)
        lib.oracle_capacity.argtypes = [_P]
        lib.oracle_capacity.restype = _I64
        lib.oracle_router_logits.argtypes = [_P, _P, _P, _P]
        lib.oracle_softmax.argtypes = [_I64, _I64, _P, _P, _P]
        lib.oracle_topk.argtypes = [_I64, _I64, _I64, _P, _P]
        lib.oracle_gates.argtypes = [_P, _P, _P, _P]
        lib.oracle_assign.argtypes = [_P, _P, _I64, _P, _P, _P, _P]
        lib.oracle_assign.restype = _I64
        lib.oracle_assign_shard.argtypes = [_P, _P, _I64, _P, _P, _P, _P, _P]
        lib.oracle_assign_shard.restype = _I64
        lib.oracle_expert_choice.argtypes = [_P, _P, _I64, _P]
        lib.oracle_stats.argtypes = [_P, _P, _P, _P, _P, _P]
        lib.oracle_expert_apply.argtypes = [_P, _P, ctypes.c_int32, _I64, _P, _P]
        lib.oracle_combine_tokens.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _I64, _P]
        lib.oracle_round_bf16.argtypes = [ctypes.c_float]
        lib.oracle_round_bf16.restype = ctypes.c_float
        lib.oracle_mx_quantize.argtypes = [_P, _I64, _P, _P]
        lib.oracle_entropy.argtypes = [_P, _I64]
        lib.oracle_entropy.restype = ctypes.c_double
        self.lib = lib
        self._keep = []

    # -- marshalling helpers -------------------------------------------------
    @staticmethod
    def _ptr(a: Optional[np.ndarray]):
        if a is None:
            return None
        assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
        return a.ctypes.data

    @staticmethod
    def config(w, mimic_bf16: bool = False, **over) -> OracleConfig:
        """OracleConfig from a Workload-like object (attributes as in ``inputs.Workload``)."""
        g = dict(n_tokens=w.n_tokens, d_model=w.d_model, d_ff=w.d_ff, n_experts=w.n_experts,
                 n_shared=w.n_shared, d_ff_shared=w.d_ff_shared, top_k=w.top_k,
                 capacity_factor=w.capacity_factor, gating=GATING[w.gating], act=ACT[w.act],
                 has_bias=int(bool(w.has_bias)), dtype=0 if w.dtype == "f32" else 1,
                 aux_alpha=w.aux_alpha, mimic_bf16=int(mimic_bf16),
                 passthrough=int(bool(getattr(w, "drop_passthrough", False))),
                 mx_act=int(getattr(w, "expert_weights", "bf16") == "mxfp8"))
        g.update(over)
        return OracleConfig(**g)

    def weights(self, tensors: Dict[str, Optional[np.ndarray]]) -> OracleWeights:
        ow = OracleWeights()
        for name, _ in OracleWeights._fields_:
            a = tensors.get(name)
            if a is not None:
                a = np.ascontiguousarray(a)
                self._keep.append(a)
            setattr(ow, name, self._ptr(a))
        return ow

    # -- the layer's steps ---------------------------------------------------
    def capacity(self, cfg: OracleConfig) -> int:
        return int(self.lib.oracle_capacity(ctypes.byref(cfg)))

    def router_logits(self, cfg, x: np.ndarray, ow: OracleWeights) -> np.ndarray:
        L = np.empty((cfg.n_tokens, cfg.n_experts), np.float32)
        self.lib.oracle_router_logits(ctypes.byref(cfg), self._ptr(np.ascontiguousarray(x)), ctypes.byref(ow),
                                      self._ptr(L))
        return L

    def softmax(self, logits: np.ndarray):
        logits = np.ascontiguousarray(logits, np.float32)
        N, E = logits.shape
        p = np.empty((N, E), np.float64)
        lse = np.empty(N, np.float64)
        self.lib.oracle_softmax(N, E, self._ptr(logits), self._ptr(p), self._ptr(lse))
        return p, lse

    def topk(self, logits: np.ndarray, k: int) -> np.ndarray:
        logits = np.ascontiguousarray(logits, np.float32)
        N, E = logits.shape
        idx = np.empty((N, k), np.int32)
        self.lib.oracle_topk(N, E, k, self._ptr(logits), self._ptr(idx))
        return idx

    def gates(self, cfg, logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
        logits = np.ascontiguousarray(logits, np.float32)
        idx = np.ascontiguousarray(idx, np.int32)
        g = np.empty(idx.shape, np.float64)
        self.lib.oracle_gates(ctypes.byref(cfg), self._ptr(logits), self._ptr(idx), self._ptr(g))
        return g

    def assign(self, cfg, idx: np.ndarray, cap: int) -> Dict[str, np.ndarray]:
        idx = np.ascontiguousarray(idx, np.int32)
        E = cfg.n_experts
        row_of = np.empty(idx.shape, np.int32)
        off = np.empty(E + 1, np.int32)
        counts = np.empty(E, np.int32)
        kept = np.empty(E, np.int32)
        dropped = self.lib.oracle_assign(ctypes.byref(cfg), self._ptr(idx), cap, self._ptr(row_of),
                                         self._ptr(off), self._ptr(counts), self._ptr(kept))
        return dict(row_of=row_of, expert_off=off, counts=counts, kept=kept, dropped=int(dropped))

    def assign_shard(self, cfg, idx: np.ndarray, cap: int, base: np.ndarray) -> Dict[str, np.ndarray]:
        """oracle_assign for one contiguous token shard whose experts already hold
        ``base[e]`` assignments from earlier tokens of the batch."""
        idx = np.ascontiguousarray(idx, np.int32)
        base = np.ascontiguousarray(base, np.int32)
        E = cfg.n_experts
        row_of = np.empty(idx.shape, np.int32)
        off = np.empty(E + 1, np.int32)
        counts = np.empty(E, np.int32)
        kept = np.empty(E, np.int32)
        dropped = self.lib.oracle_assign_shard(ctypes.byref(cfg), self._ptr(idx), cap, self._ptr(base),
                                               self._ptr(row_of), self._ptr(off), self._ptr(counts),
                                               self._ptr(kept))
        return dict(row_of=row_of, expert_off=off, counts=counts, kept=kept, dropped=int(dropped))

    def expert_choice(self, cfg, keys: np.ndarray, cap: int) -> np.ndarray:
        keys = np.ascontiguousarray(keys, np.float32)
        sel = np.empty((cfg.n_experts, cap), np.int32)
        self.lib.oracle_expert_choice(ctypes.byref(cfg), self._ptr(keys), cap, self._ptr(sel))
        return sel

    def stats(self, cfg, logits: np.ndarray, counts: np.ndarray) -> Dict[str, object]:
        logits = np.ascontiguousarray(logits, np.float32)
        counts = np.ascontiguousarray(counts, np.int32)
        E = cfg.n_experts
        f = np.empty(E, np.float64)
        P = np.empty(E, np.float64)
        out = np.empty(3, np.float64)
        self.lib.oracle_stats(ctypes.byref(cfg), self._ptr(logits), self._ptr(counts), self._ptr(f),
                              self._ptr(P), self._ptr(out))
        return dict(f=f, P=P, aux_loss=float(out[0]), z_loss=float(out[1]), mean_lse_sq=float(out[2]))

    def expert_apply(self, cfg, ow, e: int, x_row: np.ndarray, shared: bool = False) -> np.ndarray:
        x_row = np.ascontiguousarray(x_row, np.float64)
        y = np.empty(cfg.d_model, np.float64)
        self.lib.oracle_expert_apply(ctypes.byref(cfg), ctypes.byref(ow), int(shared), e, self._ptr(x_row),
                                     self._ptr(y))
        return y

    def mx_quantize(self, v: np.ndarray):
        """MXFP8 quantisation of the last axis (a multiple of 32): (E4M3 codes uint8,
        E8M0 scale bytes uint8 [..., K / 32])."""
        v = np.ascontiguousarray(v, np.float64)
        K = v.shape[-1]
        assert K % 32 == 0
        codes = np.empty(v.shape, np.uint8)
        scales = np.empty(v.shape[:-1] + (K // 32,), np.uint8)
        self.lib.oracle_mx_quantize(self._ptr(v), v.size, self._ptr(codes), self._ptr(scales))
        return codes, scales

    def round_bf16(self, v: float) -> float:
        """The mimic mode's fp32 -> bf16 rounding of one value."""
        return float(self.lib.oracle_round_bf16(float(v)))

    def entropy(self, p: Sequence[float]) -> float:
        a = np.ascontiguousarray(np.asarray(p, np.float64))
        return float(self.lib.oracle_entropy(self._ptr(a), a.size))

    # -- composition ----------------------------------------------------------
    def route(self, cfg, x: Optional[np.ndarray], ow: Optional[OracleWeights],
              logits: Optional[np.ndarray] = None, ec_keys: Optional[np.ndarray] = None) -> Dict[str, object]:
        """Routing of all N tokens. ``logits`` (fp32 [N,E]) replaces the oracle's own
        router output when given; ``ec_keys`` (fp32 [N,E]) replaces the softmax
        probabilities as expert-choice selection keys when given."""
        if logits is None:
            logits = self.router_logits(cfg, x, ow)
        logits = np.ascontiguousarray(logits, np.float32)
        cap = self.capacity(cfg)
        r: Dict[str, object] = dict(logits=logits, capacity=cap)
        if cfg.gating == 3:
            p, _ = self.softmax(logits)
            keys = ec_keys if ec_keys is not None else p.astype(np.float32)
            sel = self.expert_choice(cfg, keys, cap)
            gate_ec = np.take_along_axis(p.T, sel.astype(np.int64), axis=1)  # p[sel[e,c], e]
            r.update(sel=sel, gate_ec=np.ascontiguousarray(gate_ec), probs=p)
            counts = np.full(cfg.n_experts, cap, np.int32)
            r.update(counts=counts, dropped=0, rows=cfg.n_experts * cap)
        else:
            idx = self.topk(logits, cfg.top_k)
            g = self.gates(cfg, logits, idx)
            a = self.assign(cfg, idx, cap)
            r.update(idx=idx, gate=g, **a)
            r["rows"] = int(a["expert_off"][-1])
        r["stats"] = self.stats(cfg, logits, r["counts"])
        return r

    def outputs(self, cfg, x: np.ndarray, ow: OracleWeights, routing: Dict[str, object],
                tokens: Optional[Sequence[int]] = None) -> np.ndarray:
        """Layer output rows (fp64 [len(tokens), d]) for the listed tokens (default all)."""
        if tokens is None:
            tokens = np.arange(cfg.n_tokens, dtype=np.int64)
        tokens = np.ascontiguousarray(np.asarray(tokens, np.int64))
        out = np.empty((tokens.size, cfg.d_model), np.float64)
        x = np.ascontiguousarray(x)
        if cfg.gating == 3:
            sel = routing["sel"]
            gec = np.ascontiguousarray(routing["gate_ec"], np.float64)
            cap = int(routing["capacity"])
            self.lib.oracle_combine_tokens(ctypes.byref(cfg), self._ptr(x), ctypes.byref(ow), None, None, None,
                                           self._ptr(sel), self._ptr(gec), cap, self._ptr(tokens), tokens.size,
                                           self._ptr(out))
        else:
            idx = routing["idx"]
            g = np.ascontiguousarray(routing["gate"], np.float64)
            row_of = routing["row_of"]
            self.lib.oracle_combine_tokens(ctypes.byref(cfg), self._ptr(x), ctypes.byref(ow), self._ptr(idx),
                                           self._ptr(g), self._ptr(row_of), None, None, 0, self._ptr(tokens),
                                           tokens.size, self._ptr(out))
        return out


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    """Value of FP8 E4M3 codes (OCP 8-bit floating point, "E4M3"): sign bit, 4
    exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
    (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. fp64."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    v = np.where((e == 15) & ((c & 7) == 7), np.nan, v)
    return sign * v


_E4M3_F32 = None


def mxfp8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """OCP MX "MXFP8" weights [..., K] back to their values: E4M3 code value times
    2^(s - 127), one E8M0 scale byte s per 32 consecutive elements along K. fp32, which
    holds every such product exactly (a code has at most 4 significant bits); the code
    values come from the table e4m3_value gives for all 256 codes."""
    global _E4M3_F32
    if _E4M3_F32 is None:
        _E4M3_F32 = e4m3_value(np.arange(256, dtype=np.uint8)).astype(np.float32)
    codes = np.asarray(codes, np.uint8)
    K = codes.shape[-1]
    s = np.asarray(scales, np.uint8)
    assert s.shape[-1] * 32 == K and not np.any(s == 255)
    v = _E4M3_F32[codes].reshape(codes.shape[:-1] + (K // 32, 32))
    v *= np.exp2(s.astype(np.float32) - np.float32(127.0))[..., None]
    return v.reshape(codes.shape)


def as_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp64 values that are exactly bf16 numbers, as the oracle's bf16 bit patterns
    (asserts exactness: the dequantised MXFP8 weights have at most 4 significant bits)."""
    v = np.asarray(v)
    f = v if v.dtype == np.float32 else v.astype(np.float32)
    if v.dtype != np.float32:
        assert np.array_equal(f.astype(np.float64), v.astype(np.float64)), "not exact in fp32"
    bits = np.ascontiguousarray(f).view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "not exact in bf16"
    return np.ascontiguousarray((bits >> 16).astype(np.uint16))


def torch_to_numpy(t) -> np.ndarray:
    """A CPU copy of a torch tensor as the oracle takes it (bf16 -> uint16 bit patterns)."""
    import torch
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def weights_to_numpy(inputs: Dict[str, object]) -> Dict[str, Optional[np.ndarray]]:
    return {k: (None if v is None else torch_to_numpy(v)) for k, v in inputs.items()}
