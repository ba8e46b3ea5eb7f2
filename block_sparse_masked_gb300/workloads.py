"""Seeded synthetic inputs for the five masked-attention workloads.

This module only draws inputs: random Q/K/V, interval endpoints, block masks,
varlen sample splits and ALiBi slopes. It contains none of the method's
arithmetic (no mask expansion, no classification, no attention), so both the
CUDA path and the CPU oracle can consume exactly the same tensors.

Workloads (all bf16, head dimension d, physical tiles 128x128 on the GPU):

* ``tiny_causal``       B=1, H=2, S=256, d=64, fixed-length BSHD, causal
                        (one interval per row, F0 = q+1).
* ``sliding_sink``      B=4, H=16, S=4096, d=128, BSHD, three endpoints per
                        row: a 4-key attention sink plus a 1024-key window
                        ending at q.
* ``varlen_doc_causal`` THD, 16384 tokens in 8 documents of seeded length
                        (minimum 256), H=16, d=128, causal inside each
                        document (F0 = local q + 1).
* ``video_block_sparse`` B=1, H=24, S=32768, d=128, per-head logical block
                        mask at (B_Q, B_KV) = (64, 64), each block pair
                        active i.i.d. with probability 0.1 plus the diagonal.
* ``prefix_alibi_softcap`` B=2, H=32, S=8192, d=128, per-sample prefix
                        P ~ U[1024, 4096], F0 = max(P, q+1); score_mod is a
                        tanh softcap of 50 followed by ALiBi with slope
                        2^(-8(h+1)/32) times (k - q).
* ``decode_paged``      decoding (one query per sequence) over a paged KV
                        cache: B=32 sequences of k_len ~ U[2048, 32768],
                        Hq=32, Hk=8, d=128, 64-token pages in a random
                        permutation of the page pool, causal at the
                        query's absolute position (``decode_paged`` below).

Q/K/V are N(0, 1) draws from a seeded CPU ``torch.Generator`` rounded to
bf16; whoever consumes them (GPU path or oracle) sees the rounded values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

LAYOUT_BSHD = 0
LAYOUT_THD = 1


@dataclasses.dataclass
class Workload:
    """One synthetic problem instance.  All tensors live on the CPU."""

    name: str
    layout: int                     # LAYOUT_BSHD or LAYOUT_THD
    B: int                          # samples
    Sq: int                         # BSHD: per-sample Q length; THD: max_seqlen_q
    Sk: int                         # BSHD: per-sample K length; THD: max_seqlen_k
    Hq: int
    Hk: int
    d: int
    q: torch.Tensor                 # bf16 [B,Sq,Hq,d] or [total_q,Hq,d]
    k: torch.Tensor                 # bf16 [B,Sk,Hk,d] or [total_k,Hk,d]
    v: torch.Tensor
    scale: float
    mask_kind: str                  # "intervals" or "blocks"
    mask_func: Optional[np.ndarray] = None    # int32 [Hmask, nfunc, total_q]
    block_mask: Optional[np.ndarray] = None   # uint8 [Hmask, nbq, nbk]
    block_q: int = 0
    block_kv: int = 0
    cu_seqlens_q: Optional[np.ndarray] = None  # int32 [B+1] (THD only)
    cu_seqlens_k: Optional[np.ndarray] = None
    softcap: float = 0.0            # 0 disables the tanh softcap
    alibi_slopes: Optional[np.ndarray] = None  # float32 [Hq] or None

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0] * (self.q.shape[1] if self.layout == LAYOUT_BSHD else 1))

    @property
    def total_k(self) -> int:
        return int(self.k.shape[0] * (self.k.shape[1] if self.layout == LAYOUT_BSHD else 1))

    @property
    def Hmask(self) -> int:
        m = self.mask_func if self.mask_kind == "intervals" else self.block_mask
        return int(m.shape[0])

    def mask_only(self) -> "Workload":
        """Copy with zero-width Q/K/V (same leading shapes): cheap to pickle."""
        z = lambda t: torch.empty(tuple(t.shape[:-1]) + (0,), dtype=t.dtype)
        c = dataclasses.replace(self, q=z(self.q), k=z(self.k), v=z(self.v))
        for extra in ("prefix",):
            if hasattr(self, extra):
                setattr(c, extra, getattr(self, extra))
        return c

    def sample_bounds(self):
        """[(q_offset, q_len, k_offset, k_len)] per sample, in token rows."""
        if self.layout == LAYOUT_BSHD:
            return [(b * self.Sq, self.Sq, b * self.Sk, self.Sk) for b in range(self.B)]
        cq, ck = self.cu_seqlens_q, self.cu_seqlens_k
        return [(int(cq[b]), int(cq[b + 1] - cq[b]), int(ck[b]), int(ck[b + 1] - ck[b]))
                for b in range(self.B)]


def _qkv(gen: torch.Generator, shape_q, shape_k):
    q = torch.randn(shape_q, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(shape_k, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shape_k, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v


def _local_positions(B: int, S: int) -> np.ndarray:
    """Sample-local Q position of every flattened batch-major Q row."""
    return np.tile(np.arange(S, dtype=np.int64), B)


def tiny_causal(seed: int = 0) -> Workload:
    B, H, S, d = 1, 2, 256, 64
    gen = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(gen, (B, S, H, d), (B, S, H, d))
    qpos = _local_positions(B, S)
    mf = (qpos + 1).astype(np.int32).reshape(1, 1, B * S)
    return Workload("tiny_causal", LAYOUT_BSHD, B, S, S, H, H, d, q, k, v,
                    1.0 / math.sqrt(d), "intervals", mask_func=mf)


def causal_rows(qpos) -> np.ndarray:
    """Endpoints [1, n] of causal rows at positions qpos: F0 = q + 1."""
    return (np.asarray(qpos, np.int64) + 1).reshape(1, -1)


def sliding_sink_rows(qpos, window: int, sink: int) -> np.ndarray:
    """Endpoints [3, n] of rows at positions qpos that see a sink of `sink`
    keys and a window of `window` keys ending at q."""
    qpos = np.asarray(qpos, np.int64)
    f0 = np.minimum(sink, qpos + 1)
    f1 = np.maximum(f0, qpos - (window - 1))
    f2 = qpos + 1
    return np.stack([f0, f1, f2])


def sliding_sink(seed: int = 0, B: int = 4, H: int = 16, S: int = 4096, d: int = 128,
                 window: int = 1024, sink: int = 4) -> Workload:
    gen = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(gen, (B, S, H, d), (B, S, H, d))
    qpos = _local_positions(B, S)
    mf = sliding_sink_rows(qpos, window, sink).astype(np.int32).reshape(1, 3, B * S)
    return Workload("sliding_sink", LAYOUT_BSHD, B, S, S, H, H, d, q, k, v,
                    1.0 / math.sqrt(d), "intervals", mask_func=mf)


def doc_lengths(seed: int, total: int = 16384, ndocs: int = 8, min_len: int = 256) -> np.ndarray:
    """Seeded document lengths: min_len plus a uniform split of the rest."""
    rng = np.random.default_rng(seed)
    rest = total - ndocs * min_len
    cuts = np.sort(rng.integers(0, rest, size=ndocs - 1, endpoint=True))
    parts = np.diff(np.concatenate([[0], cuts, [rest]]))
    return (parts + min_len).astype(np.int64)


def varlen_doc_causal(seed: int = 0, total: int = 16384, ndocs: int = 8, H: int = 16,
                      d: int = 128, min_len: int = 256) -> Workload:
    lens = doc_lengths(seed, total, ndocs, min_len)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    gen = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(gen, (total, H, d), (total, H, d))
    local = np.concatenate([np.arange(n, dtype=np.int64) for n in lens])
    mf = (local + 1).astype(np.int32).reshape(1, 1, total)
    mx = int(lens.max())
    return Workload("varlen_doc_causal", LAYOUT_THD, ndocs, mx, mx, H, H, d, q, k, v,
                    1.0 / math.sqrt(d), "intervals", mask_func=mf,
                    cu_seqlens_q=cu.copy(), cu_seqlens_k=cu.copy())


def random_block_mask(seed: int, H: int, nbq: int, nbk: int, density: float = 0.1,
                      diagonal: bool = True) -> np.ndarray:
    rng = np.random.default_rng(seed)
    m = (rng.random((H, nbq, nbk)) < density).astype(np.uint8)
    if diagonal:
        n = min(nbq, nbk)
        m[:, np.arange(n), np.arange(n)] = 1
    return m


def video_block_sparse(seed: int = 0, B: int = 1, H: int = 24, S: int = 32768, d: int = 128,
                       block: int = 64, density: float = 0.1) -> Workload:
    gen = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(gen, (B, S, H, d), (B, S, H, d))
    nb = -(-S // block)
    bm = random_block_mask(seed, H, nb, nb, density)
    return Workload("video_block_sparse", LAYOUT_BSHD, B, S, S, H, H, d, q, k, v,
                    1.0 / math.sqrt(d), "blocks", block_mask=bm, block_q=block, block_kv=block)


def alibi_slopes(H: int, max_bias: float = 8.0) -> np.ndarray:
    """Per-head slopes 2^(-max_bias*(h+1)/H) as float32 (the values both sides use)."""
    return np.array([2.0 ** (-max_bias * (h + 1) / H) for h in range(H)], dtype=np.float32)


def prefix_alibi_softcap(seed: int = 0, B: int = 2, H: int = 32, S: int = 8192, d: int = 128,
                         pmin: int = 1024, pmax: int = 4096, softcap: float = 50.0) -> Workload:
    gen = torch.Generator().manual_seed(seed)
    q, k, v = _qkv(gen, (B, S, H, d), (B, S, H, d))
    rng = np.random.default_rng(seed)
    prefix = rng.integers(pmin, pmax, size=B, endpoint=True)
    qpos = _local_positions(B, S)
    pref_rows = np.repeat(prefix, S)
    mf = np.maximum(pref_rows, qpos + 1).astype(np.int32).reshape(1, 1, B * S)
    w = Workload("prefix_alibi_softcap", LAYOUT_BSHD, B, S, S, H, H, d, q, k, v,
                 1.0 / math.sqrt(d), "intervals", mask_func=mf, softcap=softcap,
                 alibi_slopes=alibi_slopes(H))
    w.prefix = prefix  # type: ignore[attr-defined]
    return w


WORKLOADS = {
    "tiny_causal": tiny_causal,
    "sliding_sink": sliding_sink,
    "varlen_doc_causal": varlen_doc_causal,
    "video_block_sparse": video_block_sparse,
    "prefix_alibi_softcap": prefix_alibi_softcap,
}


def make(name: str, seed: int = 0, **kw) -> Workload:
    return WORKLOADS[name](seed=seed, **kw)


@dataclasses.dataclass
class DecodeWorkload:
    """Decoding over a paged KV cache: q_len query rows per sequence (the
    newest tokens, at absolute positions offset_b + i with offset_b = k_len_b
    - q_len), K/V in pages of ``page_size`` tokens.  Logical key j of
    sequence b lives in page ``page_table[b, j // page_size]`` at row
    ``j % page_size``; table entries past a sequence's last page hold -1.
    Rows of a sequence's last page past k_len, and pages no sequence uses,
    hold NaN: nothing may read them.  ``mask_func`` holds the endpoints of
    each query row evaluated at its absolute position (the mask converted
    for inference)."""

    name: str
    B: int
    q_len: int
    Hq: int
    Hk: int
    d: int
    q: torch.Tensor                 # bf16 [B*q_len, Hq, d] (THD, q_len rows per sequence)
    k_cache: torch.Tensor           # bf16 [num_pages, page_size, Hk, d]
    v_cache: torch.Tensor
    page_table: np.ndarray          # int32 [B, pages_per_seq]
    page_size: int
    k_lens: np.ndarray              # int64 [B]
    mask_func: np.ndarray           # int32 [1, nfunc, B*q_len]
    scale: float
    mask_name: str = "causal"
    softcap: float = 0.0            # 0 disables the tanh softcap
    alibi_slopes: Optional[np.ndarray] = None  # float32 [Hq] or None; bias slope * (k - q_abs)

    @property
    def offsets(self) -> np.ndarray:
        return self.k_lens - self.q_len

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        return (np.arange(self.B + 1) * self.q_len).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.k_lens)]).astype(np.int32)

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])


def decode_paged(seed: int = 0, B: int = 32, Hq: int = 32, Hk: int = 8, d: int = 128,
                 page_size: int = 64, kmin: int = 2048, kmax: int = 32768, q_len: int = 1,
                 mask: str = "causal", window: int = 8192, sink: int = 4, spare_pages: int = 8,
                 k_lens=None) -> DecodeWorkload:
    rng = np.random.default_rng(seed)
    if k_lens is None:
        k_lens = rng.integers(kmin, kmax, size=B, endpoint=True)
    k_lens = np.asarray(k_lens, np.int64)
    assert np.all(k_lens >= q_len)
    npg = -(-k_lens // page_size)
    pages_per_seq = max(1, int(npg.max()))
    num_pages = int(npg.sum()) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, pages_per_seq), -1, np.int32)
    at = 0
    for b in range(B):
        table[b, :npg[b]] = perm[at:at + npg[b]]
        at += int(npg[b])
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((B * q_len, Hq, d), generator=gen).to(torch.bfloat16)
    kc = torch.randn((num_pages, page_size, Hk, d), generator=gen).to(torch.bfloat16)
    vc = torch.randn((num_pages, page_size, Hk, d), generator=gen).to(torch.bfloat16)
    used = np.zeros((num_pages, page_size), bool)
    for b in range(B):
        j = np.arange(k_lens[b])
        used[table[b, j // page_size], j % page_size] = True
    nan_rows = torch.from_numpy(~used)
    kc[nan_rows] = float("nan")
    vc[nan_rows] = float("nan")
    qpos = (np.repeat(k_lens - q_len, q_len) + np.tile(np.arange(q_len), B))
    if mask == "causal":
        mf = causal_rows(qpos)
    elif mask == "sliding":
        mf = sliding_sink_rows(qpos, window, sink)
    else:
        raise ValueError(mask)
    return DecodeWorkload("decode_paged", B, q_len, Hq, Hk, d, q, kc, vc, table, page_size, k_lens,
                          mf.astype(np.int32)[None], 1.0 / math.sqrt(d), mask)


def random_intervals(seed: int, B: int, Sq: int, Sk: int, nfunc: int, Hmask: int = 1,
                     lens_q=None, lens_k=None) -> np.ndarray:
    """Random sorted endpoints in [0, k_len] (equal neighbours included) for fuzzing.

    With ``lens_q``/``lens_k`` (varlen) each sample's rows draw endpoints in
    [0, lens_k[b]]; otherwise every row uses [0, Sk].
    """
    rng = np.random.default_rng(seed)
    if lens_q is None:
        lens_q = [Sq] * B
        lens_k = [Sk] * B
    cols = []
    for b in range(len(lens_q)):
        nq, nk = int(lens_q[b]), int(lens_k[b])
        e = rng.integers(0, nk, size=(Hmask, nfunc, nq), endpoint=True)
        # bias towards structure: snap some endpoints onto tile edges and ends
        snap = rng.random(e.shape) < 0.2
        e = np.where(snap, (e // 128) * 128, e)
        e = np.sort(e, axis=1)
        dup = rng.random(e.shape) < 0.1
        e[:, 1:, :] = np.where(dup[:, 1:, :], e[:, :-1, :], e[:, 1:, :])
        cols.append(e)
    return np.concatenate(cols, axis=2).astype(np.int32)
