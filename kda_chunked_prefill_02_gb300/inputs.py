"""Seeded synthetic inputs shaped like the KDA prefill / verify workloads.

This module holds none of the method's arithmetic: it only draws random
numbers and lays them out.  Both the CUDA path's tests and the CPU oracle are
fed from it.

Recipe (numpy PCG64, one independent stream per tensor):
  * q, k ~ N(0, 1) in fp32, L2-normalised per (token, head) in fp32, then
    rounded to bf16 (round-to-nearest-even, by torch).
  * v ~ N(0, 1) -> bf16.
  * g = -gate_bound * sigmoid(N(0, 1)) in fp32: a per-key-channel log decay in
    (-gate_bound, 0); gate_bound defaults to 5, the production gate bound of
    the cuDNN-frontend sm90 KDA page (Conversation).
  * b ~ N(0, 1) fp32: beta logits (the kernel applies the sigmoid).
  * initial state ~ N(0, init_std^2) fp32 [N, H, K, V], or None.
  * varlen lengths: one sequence of length 1 at a seeded position, the others
    uniform weights rescaled to the remaining total and clamped to
    [2, max_len], with at least three lengths that are not multiples of 64.
"""
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

HEAD_K = 128
HEAD_V = 128

# One stream id per tensor, so a tensor's values do not depend on which other
# tensors were drawn.
_Q, _K, _V, _G, _B, _S0, _LEN, _ACC, _PERM = range(9)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), stream])))


def _normal(seed, stream, shape, block=1 << 24):
    """float32 N(0,1) of `shape`, drawn in blocks to bound host memory."""
    rng = _rng(seed, stream)
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    for s in range(0, out.size, block):
        e = min(out.size, s + block)
        out[s:e] = rng.standard_normal(e - s, dtype=np.float32)
    return out.reshape(shape)


def _to_bf16(x: np.ndarray, normalize_last: bool) -> torch.Tensor:
    """fp32 numpy -> torch bf16, optionally L2-normalising the last dim in fp32.
    Processed in row blocks so huge tensors need little extra memory."""
    rows = x.reshape(-1, x.shape[-1])
    out = torch.empty(rows.shape, dtype=torch.bfloat16)
    step = 1 << 18
    for s in range(0, rows.shape[0], step):
        blk = rows[s:s + step]
        if normalize_last:
            nrm = np.sqrt(np.sum(blk * blk, axis=-1, keepdims=True, dtype=np.float32))
            blk = (blk / np.maximum(nrm, np.float32(1e-12))).astype(np.float32)
        out[s:s + step] = torch.from_numpy(np.ascontiguousarray(blk)).to(torch.bfloat16)
    return out.reshape(x.shape)


def _gate(seed, shape, gate_bound):
    z = _normal(seed, _G, shape)
    flat = z.reshape(-1)
    step = 1 << 24
    for s in range(0, flat.size, step):
        blk = flat[s:s + step]
        flat[s:s + step] = (-np.float32(gate_bound)) / (np.float32(1.0) + np.exp(-blk))
    return torch.from_numpy(z)


def varlen_lengths(seed: int, n: int, total: int, max_len: int = 8192, min_len: int = 2,
                   n_unaligned: int = 3) -> List[int]:
    """n lengths summing to `total` (one of length 1), see module docstring."""
    if n == 1:
        return [total]
    for attempt in range(1000):
        rng = _rng(seed * 1000 + attempt, _LEN)
        w = rng.uniform(0.1, 1.0, n - 1)
        rest = total - 1
        L = np.clip(np.floor(w / w.sum() * rest).astype(np.int64), min_len, max_len)
        rem = rest - int(L.sum())
        order = np.argsort(-L)
        i = 0
        while rem != 0 and i < 10 * n:
            j = order[i % (n - 1)]
            room = (max_len - L[j]) if rem > 0 else (L[j] - min_len)
            d = int(np.sign(rem)) * min(abs(rem), int(room))
            L[j] += d
            rem -= d
            i += 1
        if rem != 0:
            continue
        pos = int(rng.integers(0, n))
        lens = [int(x) for x in L]
        lens.insert(pos, 1)
        if sum(1 for x in lens if x % 64 != 0) >= n_unaligned and sum(lens) == total:
            return lens
    raise RuntimeError("could not draw varlen lengths")


def _opt(t, f):
    return None if t is None else f(t)


@dataclass
class PrefillInputs:
    q: torch.Tensor          # bf16 [B,T,H,K] (padded) or [T_total,H,K] (varlen)
    k: torch.Tensor
    v: torch.Tensor          # bf16 [..., H, V]
    g: torch.Tensor          # fp32 [..., H, K]
    beta: torch.Tensor       # fp32 [..., H] (logits)
    initial_state: Optional[torch.Tensor]   # fp32 [N,H,K,V] or None
    cu_seqlens: Optional[torch.Tensor]      # int32 [N+1] (varlen) or None (padded)
    lengths: List[int]

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)

    @property
    def num_heads(self) -> int:
        return self.q.shape[-2]

    @property
    def total_tokens(self) -> int:
        return sum(self.lengths)

    def _map(self, f):
        return PrefillInputs(f(self.q), f(self.k), f(self.v), f(self.g), f(self.beta),
                             _opt(self.initial_state, f), _opt(self.cu_seqlens, f),
                             list(self.lengths))

    def to(self, device, non_blocking=False):
        return self._map(lambda t: t.to(device, non_blocking=non_blocking))

    def pin_memory(self):
        return self._map(lambda t: t.pin_memory())


def prefill_inputs(seed: int, *, H: int, B: Optional[int] = None, T: Optional[int] = None,
                   lengths: Optional[List[int]] = None, K: int = HEAD_K, V: int = HEAD_V,
                   init_std: Optional[float] = 0.02, normalize_qk: bool = True,
                   gate_bound: float = 5.0) -> PrefillInputs:
    """Padded (B, T) or packed varlen (lengths) KDA prefill inputs."""
    if lengths is None:
        assert B is not None and T is not None
        lead, lens, cu = (B, T), [T] * B, None
    else:
        lens = [int(x) for x in lengths]
        lead = (sum(lens),)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    N = len(lens)
    q = _to_bf16(_normal(seed, _Q, lead + (H, K)), normalize_qk)
    k = _to_bf16(_normal(seed, _K, lead + (H, K)), normalize_qk)
    v = _to_bf16(_normal(seed, _V, lead + (H, V)), False)
    g = _gate(seed, lead + (H, K), gate_bound)
    beta = torch.from_numpy(_normal(seed, _B, lead + (H,)))
    s0 = None
    if init_std:
        s0 = torch.from_numpy(_normal(seed, _S0, (N, H, K, V)) * np.float32(init_std))
    return PrefillInputs(q, k, v, g, beta, s0, cu, lens)


@dataclass
class VerifyInputs:
    q: torch.Tensor          # bf16 [R,D,H,K]
    k: torch.Tensor
    v: torch.Tensor          # bf16 [R,D,H,V]
    g: torch.Tensor          # fp32 [R,D,H,K]
    beta: torch.Tensor       # fp32 [R,D,H] (logits)
    state_pool: torch.Tensor  # fp32 [P,H,K,V]
    accepted: torch.Tensor   # int32 [R] in 0..D
    slot: Optional[torch.Tensor]  # int32 [R] or None (= r)

    def to(self, device, non_blocking=False):
        f = (lambda t: t.to(device, non_blocking=non_blocking))
        return VerifyInputs(f(self.q), f(self.k), f(self.v), f(self.g), f(self.beta),
                            f(self.state_pool), f(self.accepted), _opt(self.slot, f))


def verify_inputs(seed: int, *, R: int, D: int, H: int, K: int = HEAD_K, V: int = HEAD_V,
                  pool_size: Optional[int] = None, permute_slots: bool = False,
                  init_std: float = 0.02, gate_bound: float = 5.0) -> VerifyInputs:
    lead = (R, D)
    q = _to_bf16(_normal(seed, _Q, lead + (H, K)), True)
    k = _to_bf16(_normal(seed, _K, lead + (H, K)), True)
    v = _to_bf16(_normal(seed, _V, lead + (H, V)), False)
    g = _gate(seed, lead + (H, K), gate_bound)
    beta = torch.from_numpy(_normal(seed, _B, lead + (H,)))
    P = pool_size or R
    pool = torch.from_numpy(_normal(seed, _S0, (P, H, K, V)) * np.float32(init_std))
    acc = torch.from_numpy(_rng(seed, _ACC).integers(0, D + 1, R).astype(np.int32))
    slot = None
    if permute_slots:
        slot = torch.from_numpy(_rng(seed, _PERM).permutation(P)[:R].astype(np.int32))
    return VerifyInputs(q, k, v, g, beta, pool, acc, slot)


CONFIG_DESCRIPTIONS = {
    "tiny": "B=1 T=256 H=2 K=V=128 chunk=64, zero initial state (seed 0)",
    "padded": "B=4 T=4096 H=16 K=V=128 chunk=64, initial state N(0,0.02^2) (seed 1)",
    "varlen": "8 packed sequences (one of length 1) summing to 32768 tokens, H=32 (seed 2)",
    "long": "B=1 T=131072 H=32 K=V=128 chunk=64, initial state N(0,0.02^2) (seed 3)",
    "verify": "256 requests x 4 drafts, H=32, fp32 state pool N(0,0.02^2), accepted U{0..4} (seed 4)",
    "long_h8": "B=1 T=131072 H=8 K=V=128 chunk=64, initial state N(0,0.02^2) (seed 5): the long "
               "workload with few chains",
}


def config_inputs(name: str):
    """The five workloads, seeds 0..4, and the few-chain long workload (seed 5)."""
    if name == "tiny":
        return prefill_inputs(0, B=1, T=256, H=2, init_std=None)
    if name == "padded":
        return prefill_inputs(1, B=4, T=4096, H=16)
    if name == "varlen":
        return prefill_inputs(2, lengths=varlen_lengths(2, 8, 32768), H=32)
    if name == "long":
        return prefill_inputs(3, B=1, T=131072, H=32)
    if name == "verify":
        return verify_inputs(4, R=256, D=4, H=32)
    if name == "long_h8":
        return prefill_inputs(5, B=1, T=131072, H=8)
    raise KeyError(name)


def prefix_sample(inp: PrefillInputs, max_tokens: int) -> PrefillInputs:
    """The first `max_tokens` tokens of every sequence (all heads), repacked the
    same way; used to time bounded samples of a workload."""
    if inp.cu_seqlens is None:
        m = min(max_tokens, inp.q.shape[1])
        f = lambda t: t[:, :m].contiguous()
        return PrefillInputs(f(inp.q), f(inp.k), f(inp.v), f(inp.g), f(inp.beta),
                             inp.initial_state, None, [m] * inp.q.shape[0])
    cu = inp.cu_seqlens.tolist()
    idx, lens = [], []
    for n in range(len(cu) - 1):
        m = min(max_tokens, cu[n + 1] - cu[n])
        idx.extend(range(cu[n], cu[n] + m))
        lens.append(m)
    ix = torch.tensor(idx, dtype=torch.long)
    f = lambda t: t.index_select(0, ix).contiguous()
    new_cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    return PrefillInputs(f(inp.q), f(inp.k), f(inp.v), f(inp.g), f(inp.beta),
                         inp.initial_state, new_cu, lens)
