"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws bytes and numbers; it holds none of the method's arithmetic
(no decoding of any block format). It knows only where each format keeps its
f16 scale fields, so that it can overwrite them with a bounded distribution --
the same idea as the Vulkore quant_test.cpp harness's `random_blocks`, which
fills blocks with random bytes and then bounds their scale fields.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), counter-based, so any slice can be regenerated.
Seeds follow `seed = 20260000 + 100 * config + kind_index`.

Workloads (shapes and distributions of the pages' benchmarks):
  * tiny Q4_0 qgemm           M=256,  K=1024, N=4, fp32 x ~ N(0,1), d ~ U[1e-3,1e-2]
  * decode GEMV               M=14336, K=4096, N=1, Q8_0 (int8 ~ U{-127..127}) and Q4_0
  * K-quant prefill GEMM      M=K=4096, N=512, f16 X ~ N(0,1), random bytes,
                              f16 scale fields ~ U[1e-4,1e-2]
  * codebook GEMM             M=11008, K=4096, N=128, f16 X ~ N(0,1); IQ4_NL/IQ4_XS
                              d ~ U[1e-3,1e-2]; MXFP4 E8M0 ~ U{118..130}
  * Q4_1 / Q5_1 / Q8_1 GEMM   the codebook shape (no workload on the pages), f16 X,
                              d and m ~ U[1e-3,1e-2]
  * MoE expert-grouped Q4_0   128 experts, gate_up 1536x2048, down 2048x768,
                              T in {1, 8, 64} tokens, 8 distinct experts per token
"""
from __future__ import annotations

import numpy as np

KINDS = ["Q8_0", "Q4_0", "Q5_0", "Q4_K", "Q5_K", "Q6_K",
         "Q2_K", "Q3_K", "IQ4_NL", "IQ4_XS", "MXFP4", "Q4_1", "Q5_1", "Q8_1"]
KIND_INDEX = {k: i for i, k in enumerate(KINDS)}

# (block bytes, block elements, byte offsets of the f16 scale fields)
_LAYOUT = {
    "Q8_0": (34, 32, (0,)),
    "Q4_0": (18, 32, (0,)),
    "Q5_0": (22, 32, (0,)),
    "Q4_K": (144, 256, (0, 2)),
    "Q5_K": (176, 256, (0, 2)),
    "Q6_K": (210, 256, (208,)),
    "Q2_K": (84, 256, (80, 82)),
    "Q3_K": (110, 256, (108,)),
    "IQ4_NL": (18, 32, (0,)),
    "IQ4_XS": (136, 256, (0,)),
    "MXFP4": (17, 32, ()),
    "Q4_1": (20, 32, (0, 2)),
    "Q5_1": (24, 32, (0, 2)),
    "Q8_1": (36, 32, (0,)),   # the f16 at byte 2 stays random: no element reads it
}

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def block_geometry(kind: str):
    bb, be, _ = _LAYOUT[kind]
    return bb, be


def row_bytes(kind: str, K: int) -> int:
    bb, be, _ = _LAYOUT[kind]
    if K % be:
        raise ValueError(f"K={K} is not a multiple of {kind}'s {be}-element block")
    return (K // be) * bb


def config_seed(config: int, kind: str) -> int:
    return 20260000 + 100 * config + KIND_INDEX[kind]


def _mix_inplace(z: np.ndarray, t: np.ndarray) -> None:
    """splitmix64 output function applied in place (t is scratch of z's size)."""
    np.right_shift(z, np.uint64(30), out=t)
    np.bitwise_xor(z, t, out=z)
    np.multiply(z, _M1, out=z)
    np.right_shift(z, np.uint64(27), out=t)
    np.bitwise_xor(z, t, out=z)
    np.multiply(z, _M2, out=z)
    np.right_shift(z, np.uint64(31), out=t)
    np.bitwise_xor(z, t, out=z)


_CHUNK = 1 << 22


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n outputs of splitmix64 started at `seed`, skipping the first `offset`.

    Computed in place, chunk by chunk (fresh large temporaries are slow to
    fault in)."""
    out = np.empty(n, dtype=np.uint64)
    base = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for c0 in range(0, n, _CHUNK):
            c1 = min(n, c0 + _CHUNK)
            z = out[c0:c1]
            z[:] = np.arange(offset + c0 + 1, offset + c1 + 1, dtype=np.uint64)
            np.multiply(z, _GOLDEN, out=z)
            np.add(z, base, out=z)
            _mix_inplace(z, np.empty_like(z))
    return out


def substream(seed: int, tag: int) -> int:
    """Independent seed for sub-stream `tag` of `seed`."""
    return int(splitmix64((seed * 0x100000001B3 + tag) & 0xFFFFFFFFFFFFFFFF, 1)[0])


class Stream:
    """Draws from one splitmix64 sequence (consumed in order)."""

    def __init__(self, seed: int):
        self.seed = seed & 0xFFFFFFFFFFFFFFFF
        self.pos = 0

    def u64(self, n: int) -> np.ndarray:
        out = splitmix64(self.seed, n, self.pos)
        self.pos += n
        return out

    def bytes(self, n: int) -> np.ndarray:
        words = self.u64((n + 7) // 8)
        return words.view(np.uint8)[:n].copy()

    def uniform(self, n: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
        u = (self.u64(n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        return lo + (hi - lo) * u

    def normal(self, n: int) -> np.ndarray:
        """Box-Muller, float64."""
        u1 = 1.0 - self.uniform(n)          # (0, 1]
        u2 = self.uniform(n)
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    def randint(self, n: int, lo: int, hi: int) -> np.ndarray:
        """Integers uniform on [lo, hi] (inclusive).

        Spans below 256 draw from 16-bit lanes of the generator (four per
        output word; modulo bias below 0.4 %), wider spans from whole words."""
        span = hi - lo + 1
        if span <= 256:
            lanes = self.u64((n + 3) // 4).view(np.uint16)[:n]
            return (lanes % np.uint16(span)).astype(np.int16).astype(np.int64) + lo
        return (self.u64(n) % np.uint64(span)).astype(np.int64) + lo


def f16_bits(values: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest binary16 (ties to even); return the bits."""
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def quant_weights(kind: str, rows: int, K: int, seed: int,
                  scale_lo: float = 1e-3, scale_hi: float = 1e-2,
                  e8m0_lo: int = 118, e8m0_hi: int = 130,
                  int8_codes: bool = False) -> np.ndarray:
    """rows x row_bytes bytes of `kind` blocks, flat uint8.

    Everything is uniform random bytes, except: every f16 scale field is drawn
    uniform on [scale_lo, scale_hi] and rounded to f16; the MXFP4 E8M0 byte is
    uniform on {e8m0_lo..e8m0_hi}; with int8_codes, Q8_0 codes are uniform on
    {-127..127}.
    """
    bb, be, offs = _LAYOUT[kind]
    nblk = rows * (K // be)
    if K % be:
        raise ValueError(f"K={K} is not a multiple of {be}")
    s_bytes = Stream(substream(seed, 1))
    raw = s_bytes.bytes(nblk * bb).reshape(nblk, bb)
    if kind == "Q8_0" and int8_codes:
        codes = Stream(substream(seed, 2)).randint(nblk * 32, -127, 127)
        raw[:, 2:34] = codes.astype(np.int8).view(np.uint8).reshape(nblk, 32)
    if offs:
        sc = Stream(substream(seed, 3)).uniform(nblk * len(offs), scale_lo, scale_hi)
        bits = f16_bits(sc).reshape(nblk, len(offs))
        for j, o in enumerate(offs):
            raw[:, o] = (bits[:, j] & 0xFF).astype(np.uint8)
            raw[:, o + 1] = (bits[:, j] >> 8).astype(np.uint8)
    if kind == "MXFP4":
        raw[:, 0] = Stream(substream(seed, 4)).randint(nblk, e8m0_lo, e8m0_hi).astype(np.uint8)
    return raw.reshape(-1)


def activations(n: int, K: int, seed: int, dtype: str = "f32") -> np.ndarray:
    """n x K activations ~ N(0,1), as float32 or float16 (round to nearest even)."""
    z = Stream(substream(seed, 5)).normal(n * K).reshape(n, K)
    return z.astype(np.float16 if dtype == "f16" else np.float32)


def routing(n_tokens: int, n_experts: int, top_k: int, seed: int) -> np.ndarray:
    """(n_tokens, top_k) distinct experts per token, by a seeded partial Fisher-Yates."""
    s = Stream(substream(seed, 6))
    out = np.empty((n_tokens, top_k), dtype=np.int32)
    for t in range(n_tokens):
        perm = np.arange(n_experts, dtype=np.int32)
        draws = s.u64(top_k)
        for i in range(top_k):
            j = i + int(draws[i] % np.uint64(n_experts - i))
            perm[i], perm[j] = perm[j], perm[i]
        out[t] = perm[:top_k]
    return out


# ---------------------------------------------------------------------------
# The pages' workloads
# ---------------------------------------------------------------------------
TINY = dict(config=0, kind="Q4_0", M=256, K=1024, N=4, x_dtype="f32")
DECODE = dict(config=1, kinds=("Q8_0", "Q4_0"), M=14336, K=4096, N=1, x_dtype="f32")
KQUANT = dict(config=2, kinds=("Q4_K", "Q5_K", "Q6_K", "Q2_K", "Q3_K"),
              M=4096, K=4096, N=512, x_dtype="f16", scale_lo=1e-4, scale_hi=1e-2)
CODEBOOK = dict(config=3, kinds=("IQ4_NL", "IQ4_XS", "MXFP4"),
                M=11008, K=4096, N=128, x_dtype="f16")
# Q4_1 / Q5_1 / Q8_1 have no workload on the pages: their GEMM tests take the
# codebook workload's shape.
LEGACY1 = dict(config=5, kinds=("Q4_1", "Q5_1", "Q8_1"), M=11008, K=4096, N=128, x_dtype="f16")
MOE = dict(config=4, kind="Q4_0", n_experts=128, top_k=8, d_model=2048, d_ff=768,
           tokens=(1, 8, 64), x_dtype="f32")


def workload_weights(cfg: dict, kind: str, M: int = None, K: int = None) -> np.ndarray:
    seed = config_seed(cfg["config"], kind)
    M = cfg["M"] if M is None else M
    K = cfg["K"] if K is None else K
    return quant_weights(kind, M, K, seed,
                         scale_lo=cfg.get("scale_lo", 1e-3), scale_hi=cfg.get("scale_hi", 1e-2),
                         int8_codes=(kind == "Q8_0"))


def workload_x(cfg: dict, kind: str, N: int = None, K: int = None) -> np.ndarray:
    seed = config_seed(cfg["config"], kind)
    return activations(cfg["N"] if N is None else N, cfg["K"] if K is None else K,
                       seed, cfg["x_dtype"])


def moe_problem(T: int, which: str = "gate_up", seed: int = None):
    """Weights for all experts (flat), expert stride, x, x_row, expert_id, M, K."""
    cfg = MOE
    kind = cfg["kind"]
    seed = config_seed(4, kind) + 1000 * T if seed is None else seed
    E, top = cfg["n_experts"], cfg["top_k"]
    if which == "gate_up":
        M, K = 2 * cfg["d_ff"], cfg["d_model"]
    else:
        M, K = cfg["d_model"], cfg["d_ff"]
    stride = M * row_bytes(kind, K)
    w = quant_weights(kind, E * M, K, config_seed(4, kind) + (0 if which == "gate_up" else 7))
    route = routing(T, E, top, seed)
    expert_id = route.reshape(-1).astype(np.int32)
    if which == "gate_up":
        x = activations(T, K, seed, "f32")
        x_row = np.repeat(np.arange(T, dtype=np.int32), top)
    else:
        x = activations(T * top, K, seed + 17, "f32")
        x_row = np.arange(T * top, dtype=np.int32)
    return dict(kind=kind, w=w, stride=stride, n_experts=E, x=x, x_row=x_row,
                expert_id=expert_id, M=M, K=K)


def moe_layer_problem(T: int, seed: int = None):
    """One MoE layer of the config-4 shape: both projections' weights for all
    experts, fp32 tokens, per-token top-k expert ids (distinct, seeded) and
    routing weights (uniform draws normalised to sum to one per token)."""
    cfg = MOE
    kind, E, k = cfg["kind"], cfg["n_experts"], cfg["top_k"]
    dm, dff = cfg["d_model"], cfg["d_ff"]
    seed = config_seed(4, kind) + 5000 + T if seed is None else seed
    w_gu = quant_weights(kind, E * 2 * dff, dm, config_seed(4, kind))
    w_dn = quant_weights(kind, E * dm, dff, config_seed(4, kind) + 7)
    ids = routing(T, E, k, seed)
    wt = Stream(substream(seed, 8)).uniform(T * k, 0.05, 1.0).reshape(T, k)
    wt = (wt / wt.sum(axis=1, keepdims=True)).astype(np.float32)
    x = activations(T, dm, seed + 3, "f32")
    return dict(kind=kind, w_gu=w_gu, gu_stride=2 * dff * row_bytes(kind, dm), w_down=w_dn,
                down_stride=dm * row_bytes(kind, dff), n_experts=E, x=x, ids=ids, w=wt, d_model=dm, d_ff=dff)
