"""The entry-sharded decode's exchange on CPU: world size 2 with the gloo backend, every rank one
shard of each sequence's entries. The per-shard steps are the fp64 oracle's (the kernels need a
GPU); the partition, the all-gathers of candidates and partial outputs, the global selection
from the gathered candidates and the log-sum-exp merge are the library's sharded driver
(long_context_compressed_pooling_b300.sharded.decode_step). Every rank must end with the
unsharded oracle's top-k list and output."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The per-shard steps with the fp64 oracle, on CPU tensors (test infrastructure)."""

    @staticmethod
    def candidates(sh, q_pos0, m, k):
        import oracle as O
        B, E = sh.ki_codes.shape[0], sh.ki_codes.shape[1]
        idx = np.full((B, k), -1, np.int32)
        sc = np.zeros((B, k), np.uint16)
        cnt = np.zeros(B, np.int32)
        for b in range(B):
            nv = O.visible_entries(q_pos0, m, E)
            s = O.f64_to_bf16_rne(O.index_scores(sh.qi_codes[b, 0].numpy(), sh.qi_scales[b, 0].numpy(),
                                                 sh.ki_codes[b, :nv].numpy(),
                                                 sh.ki_scales[b, :nv].numpy(), 64))
            i, c = O.topk_select(s, nv, k)
            idx[b] = i
            cnt[b] = c
            sc[b, :c] = s[i[:c]]
        return (torch.from_numpy(idx), torch.from_numpy(sc.view(np.int16)).view(torch.bfloat16),
                torch.from_numpy(cnt))

    @staticmethod
    def merge(cand_sc, cand_idx, cand_cnt, bases):
        import oracle as O
        S, B, k = cand_idx.shape
        vals = O.bf16_to_f64(cand_sc.view(torch.int16).numpy().view(np.uint16))
        topk = np.full((B, k), -1, np.int32)
        cnt = np.zeros(B, np.int32)
        sidx = np.full((S, B, k), -1, np.int32)
        scnt = np.zeros((S, B), np.int32)
        for b in range(B):
            pos, glob, vv = [], [], []
            for s in range(S):
                for j in range(int(cand_cnt[s, b])):
                    pos.append((s, int(cand_idx[s, b, j])))
                    glob.append(bases[s] + int(cand_idx[s, b, j]))
                    vv.append(vals[s, b, j])
            order = np.argsort(np.array(glob, np.int64), kind="stable")
            vv = np.array(vv)[order]
            sel, c = O.topk_select_values(vv, len(vv), k)
            cnt[b] = c
            for r, p in enumerate(sel[:c]):
                s, loc = pos[order[p]]
                topk[b, r] = bases[s] + loc
                sidx[s, b, scnt[s, b]] = loc
                scnt[s, b] += 1
        return (torch.from_numpy(topk), torch.from_numpy(cnt), torch.from_numpy(sidx),
                torch.from_numpy(scnt))

    @staticmethod
    def attend(sh, idx, cnt, t, W):
        import oracle as O
        B = idx.shape[0]
        H, d = sh.q.shape[2], sh.q.shape[3]
        out = np.zeros((B, 1, H, d))
        lse = np.zeros((B, 1, H))
        for b in range(B):
            kr = sh.k_raw[b].numpy() if sh.k_raw is not None else np.zeros((1, d))
            vr = sh.v_raw[b].numpy() if sh.v_raw is not None else np.zeros((1, d))
            o, l = O.csa_attend_one(sh.q[b, 0].numpy(), sh.k_cmp[b].numpy(), sh.v_cmp[b].numpy(),
                                    idx[b].numpy(), int(cnt[b]), kr, vr, t if W > 0 else 0, W)
            out[b, 0], lse[b, 0] = o, l
        return torch.from_numpy(out), torch.from_numpy(lse)

    @staticmethod
    def lse_merge(parts, lses):
        p, l = parts.numpy(), lses.numpy()
        L = np.max(l, axis=0)
        w = np.where(np.isneginf(l), 0.0, np.exp(l - np.where(np.isneginf(L), 0.0, L)))
        ws = w.sum(axis=0)
        out = (w[..., None] * p).sum(axis=0) / np.where(ws > 0, ws, 1.0)[..., None]
        lse = np.where(ws > 0, np.where(np.isneginf(L), 0.0, L) + np.log(np.where(ws > 0, ws, 1.0)),
                       -np.inf)
        return torch.from_numpy(out), torch.from_numpy(lse)


def _inputs(seed=5, B=2, N=2048, m=4, H=8, d=64):
    """Deterministic inputs of one layer, the same on every rank (entries pooled by the oracle)."""
    import oracle as O
    from synth import LayerShape, generate_layer
    s = LayerShape("csa", B=B, N=N, Nq=1, q_pos0=N - 1, H=H, d=d, m=m, W=16, k=40, H_I=4, d_I=64,
                   q_scale=1.0 / np.sqrt(d), compress_begin=0)
    x = generate_layer(s, seed=seed, device="cpu")
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    kr = np.stack([O.bf16_to_f64(bits(x["k_raw"][b])) for b in range(B)])
    vr = np.stack([O.bf16_to_f64(bits(x["v_raw"][b])) for b in range(B)])
    w = x["logits"].numpy().astype(np.float64)
    kc = np.stack([O.compress(kr[b], w[b], m) for b in range(B)])
    vc = np.stack([O.compress(vr[b], w[b], m) for b in range(B)])
    q = np.stack([O.bf16_to_f64(bits(x["q"][b])) for b in range(B)])
    return s, x, q, kr, vr, kc, vc


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        from long_context_compressed_pooling_b300 import sharded
        s, x, q, kr, vr, kc, vc = _inputs()
        E = s.N // s.m
        cuts = [0, 200, E]  # uneven: rank 0 the oldest 200 entries, rank 1 the rest + window
        a, e = cuts[rank], cuts[rank + 1]
        last = rank == world - 1
        sh = sharded.Shard(base=a, qi_codes=x["qi_codes"], qi_scales=x["qi_scales"],
                           ki_codes=x["ki_codes"][:, a:e], ki_scales=x["ki_scales"][:, a:e],
                           k_cmp=torch.from_numpy(kc[:, a:e]), v_cmp=torch.from_numpy(vc[:, a:e]),
                           q=torch.from_numpy(q),
                           k_raw=torch.from_numpy(kr) if last else None,
                           v_raw=torch.from_numpy(vr) if last else None)
        idx, cnt, o, l = sharded.decode_step([sh], s.q_pos0, s.m, s.k, s.W, ops=OracleOps,
                                             gather=sharded.Exchange())
        # the unsharded oracle
        bad = []
        for b in range(s.B):
            sc = O.f64_to_bf16_rne(O.index_scores(x["qi_codes"][b, 0].numpy(),
                                                  x["qi_scales"][b, 0].numpy(),
                                                  x["ki_codes"][b].numpy(),
                                                  x["ki_scales"][b].numpy(), 64))
            ridx, rcnt = O.topk_select(sc, E, s.k)
            ro, rl = O.csa_attend_one(q[b, 0], kc[b], vc[b], ridx, rcnt, kr[b], vr[b], s.q_pos0, s.W)
            if not np.array_equal(idx[b].numpy(), ridx) or int(cnt[b]) != rcnt:
                bad.append(("topk", b))
            if np.max(np.abs(o[b].numpy() - ro)) > 1e-9 or np.max(np.abs(l[b].numpy() - rl)) > 1e-9:
                bad.append(("out", b))
        out[rank] = bad
    finally:
        dist.destroy_process_group()


def test_two_rank_sharded_decode_equals_unsharded_oracle():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res == {0: [], 1: []}, res
