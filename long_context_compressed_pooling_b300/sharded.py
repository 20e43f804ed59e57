"""Entry-sharded CSA decode: the compressed entries of each sequence split over S shards.

The pages' 1M-token context (9fzt.com DeepSeek-V4 summary, item 1) makes one sequence's entry
cache worth splitting over GPUs; the CSA step (Lighthouse "deep deepseek v4 release" 八.3) then
runs as:
  1. every shard selects its own top-k candidates (csa_shard_candidates: the indexer and the
     selector over the shard's entries, with the global visibility);
  2. the candidates (local index, BF16 score, count) of all shards are exchanged;
  3. every process merges them into the global top-k (csa_topk_merge: score descending, ties to
     the lower global index, exactly the unsharded selection) and each shard's part of it;
  4. every shard attends to its part (the shard holding the newest tokens also to the window),
     returning its normalised output and log-sum-exp;
  5. the partial outputs are exchanged and merged by log-sum-exp (csa_lse_merge).

The exchange is the only collective on the data path. `decode_step` takes the shards this
process holds (one per rank under torch.distributed, or all S of them on one GPU: "virtual"
shards), the operations of steps 1, 3, 4 and 5 (`LibraryOps` runs the library's kernels on the
GPU), and a gather that returns a list over all S shards in order (`Exchange`).
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence

import torch

from . import _native as N


@dataclasses.dataclass
class Shard:
    """One shard of a CSA decode layer: entries [base, base + E_s) of every sequence."""
    base: int                  # first global entry index of the shard
    qi_codes: torch.Tensor     # [B, 1, H_I, d_I/2]   (every shard holds the index queries)
    qi_scales: torch.Tensor    # [B, 1, H_I, d_I/32]
    ki_codes: torch.Tensor     # [B, E_s, d_I/2]
    ki_scales: torch.Tensor    # [B, E_s, d_I/32]
    k_cmp: torch.Tensor        # [B, E_s, d]
    v_cmp: torch.Tensor        # [B, E_s, d]
    q: torch.Tensor            # [B, 1, H, d]         (every shard holds the queries)
    k_raw: Optional[torch.Tensor] = None  # [B, N, d] raw rows: the window's shard only
    v_raw: Optional[torch.Tensor] = None


class LibraryOps:
    """Steps 1, 3, 4, 5 on the GPU through the library's C ABI."""

    @staticmethod
    def candidates(sh: Shard, q_pos0: int, m: int, k: int):
        return N.shard_candidates(sh.qi_codes, sh.qi_scales, sh.ki_codes, sh.ki_scales, q_pos0, m, k)

    @staticmethod
    def merge(cand_scores, cand_idx, cand_cnt, bases):
        return N.topk_merge(cand_scores, cand_idx, cand_cnt, bases)

    @staticmethod
    def attend(sh: Shard, idx, cnt, t: int, W: int):
        k_raw = sh.k_raw if sh.k_raw is not None else sh.k_cmp
        v_raw = sh.v_raw if sh.v_raw is not None else sh.v_cmp
        B = idx.shape[0]
        return N.csa_attend(sh.q, sh.k_cmp, sh.v_cmp, idx.view(B, 1, -1), cnt.view(B, 1), k_raw,
                            v_raw, W, t if W > 0 else k_raw.shape[1] - 1, want_lse=True)

    @staticmethod
    def lse_merge(parts, lses):
        return N.lse_merge(parts, lses, want_lse=True)


class Exchange:
    """Gathers per-shard tensors into a list over all S shards, in shard order.

    group=None and world 1: the process holds every shard (the list is returned as it is).
    Otherwise every rank holds one shard (rank r = shard r) and the tensors are all-gathered
    through torch.distributed (as bytes, whatever their dtype)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist if dist.is_available() and dist.is_initialized() else None
        self.group = group
        self.world = self.dist.get_world_size(group) if self.dist else 1

    def __call__(self, local: Sequence[torch.Tensor]) -> List[torch.Tensor]:
        if self.world == 1:
            return list(local)
        assert len(local) == 1, "one shard per rank"
        t = local[0].contiguous()
        wire = t.view(torch.uint8)  # every dtype travels as its bytes
        out = [torch.empty_like(wire) for _ in range(self.world)]
        self.dist.all_gather(out, wire, group=self.group)
        return [o.view(t.dtype) for o in out]


def decode_step(shards: Sequence[Shard], t: int, m: int, k: int, W: int, ops=LibraryOps,
                gather: Optional[Callable] = None, window_shard: Optional[int] = None):
    """One CSA decode step of one query per sequence at position t over sharded entries.

    shards: the shards this process holds, in order (all S, or this rank's one); the shard
    index of shards[i] is i (one process) or the rank. window_shard: the shard that attends to
    the window (default: the last). Returns (topk_idx [B, k] global, topk_cnt [B], out [B, H, d],
    lse [B, H]) - the same on every process."""
    gather = gather or Exchange()
    world = getattr(gather, "world", 1)
    S = len(shards) if world == 1 else world
    first = 0 if world == 1 else gather.dist.get_rank(gather.group)
    window_shard = S - 1 if window_shard is None else window_shard
    # 1. candidates of the local shards (visibility is the global one: t relative to the shard)
    local = [ops.candidates(sh, t - sh.base * m, m, k) for sh in shards]
    # 2. exchange
    cand_idx = torch.stack(gather([c[0] for c in local]))      # [S, B, k]
    cand_sc = torch.stack(gather([c[1] for c in local]))       # [S, B, k]
    cand_cnt = torch.stack(gather([c[2] for c in local]))      # [S, B]
    bases_t = torch.stack(gather([torch.tensor([sh.base], dtype=torch.int64,
                                               device=shards[0].ki_codes.device)
                                  for sh in shards]))
    bases = [int(x) for x in bases_t.view(-1).tolist()]
    # 3. the global selection and every shard's part of it
    topk_idx, topk_cnt, shard_idx, shard_cnt = ops.merge(cand_sc, cand_idx, cand_cnt, bases)
    # 4. each local shard attends to its part (the window on one shard only)
    outs, lses = [], []
    for i, sh in enumerate(shards):
        s = first + i
        o, l = ops.attend(sh, shard_idx[s], shard_cnt[s], t, W if s == window_shard else 0)
        outs.append(o.view(o.shape[0], o.shape[-2], o.shape[-1]))
        lses.append(l.view(l.shape[0], l.shape[-1]))
    # 5. exchange and merge the partial outputs
    parts = torch.stack(gather(outs))                           # [S, B, H, d]
    parts_lse = torch.stack(gather(lses))                       # [S, B, H]
    out, lse = ops.lse_merge(parts, parts_lse)
    return topk_idx, topk_cnt, out, lse
