"""Token-tree workloads and the element-by-element comparison of the CUDA tree
verifier with the float64 oracle.

Tolerances (as for the chain verifier, tests/parity.py):
  - greedy requests: bit-exact (path, emitted token, last node);
  - sampling requests: every child both walks tested must get the same
    decision, except where the float64 oracle sits on a near-tie
    |u - r(x)/q(x)| < 1e-6; the emitted token must be identical, except where
    the emission uniform lies within 1e-6 of the GPU token's oracle CDF
    interval.  Such cases are counted ("excused"); anything else fails.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle

TIE = 1e-6


@dataclass
class TreeWorkload:
    logits: torch.Tensor   # [B, N, V] f32 | bf16 (cuda)
    probs: torch.Tensor    # [B, N, V] f32
    tokens: torch.Tensor   # [B, N] int32
    parents: torch.Tensor  # [B, N] int32
    nodes: torch.Tensor    # [B] int32
    temp: torch.Tensor     # [B] f32
    seed: int

    def to_numpy(self) -> dict:
        tl = self.logits.detach().cpu()
        tl_np = tl.view(torch.int16).numpy().view("uint16") if tl.dtype == torch.bfloat16 \
            else tl.numpy()
        return {"target_logits": tl_np, "draft_probs": self.probs.cpu().numpy(),
                "tree_tokens": self.tokens.cpu().numpy(), "tree_parents": self.parents.cpu().numpy(),
                "num_nodes": self.nodes.cpu().numpy(), "temperature": self.temp.cpu().numpy(),
                "seed": self.seed}


def random_parents(rng, B: int, N: int, width: float) -> np.ndarray:
    """Tries whose node c picks its parent among the earlier nodes; `width`
    in (0, 1] biases towards recent nodes (deep, narrow) when small."""
    par = np.full((B, N), -1, np.int32)
    for c in range(1, N):
        lo = np.maximum(0, c - np.maximum(1, (width * c)).astype(int))
        par[:, c] = rng.integers(lo, c)
    return par


def make_tree_workload(B, N, V, *, bf16=True, seed=0, greedy_frac=0.3, width=0.6,
                       noise=1.0, device="cuda") -> TreeWorkload:
    """Zipf-like target logits per node, drafts drawn from a noisy copy of the
    parent's distribution (so that many are accepted), random tries."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    rng = np.random.default_rng(seed)
    rank = torch.arange(1, V + 1, dtype=torch.float32)
    base = -1.1 * torch.log(rank)
    perm = torch.argsort(torch.rand(B, N, V, generator=g), dim=-1)
    logits = base[perm] + torch.randn(B, N, V, generator=g)
    par = random_parents(rng, B, N, width)
    T = torch.from_numpy(np.where(rng.random(B) < greedy_frac, 0.0,
                                  rng.uniform(0.5, 1.3, B)).astype(np.float32))
    # draft distribution of node c: a noisy copy of its parent's target row
    pl = logits[torch.arange(B)[:, None], torch.from_numpy(par.clip(min=0)).long()]
    dlog = pl + noise * torch.randn(B, N, V, generator=g)
    Tq = torch.where(T > 0, T, torch.ones_like(T))[:, None, None]
    q = torch.softmax(dlog / Tq, dim=-1)
    tok = torch.multinomial(q.reshape(B * N, V), 1, generator=g).reshape(B, N).to(torch.int32)
    # greedy requests: a child often repeats the parent's argmax
    am = logits.argmax(-1)
    for b in np.nonzero(T.numpy() == 0)[0]:
        for c in range(1, N):
            if rng.random() < 0.5:
                tok[b, c] = int(am[b, par[b, c]])
    tok[:, 0] = 0
    nodes = torch.from_numpy(rng.integers(1, N + 1, B).astype(np.int32))
    lt = logits.to(torch.bfloat16) if bf16 else logits
    return TreeWorkload(lt.to(device).contiguous(), q.to(device).contiguous(),
                        tok.to(device).contiguous(), torch.from_numpy(par).to(device).contiguous(),
                        nodes.to(device), T.to(device), seed * 7919 + 13)


@dataclass
class TreeReport:
    requests: int = 0
    greedy: int = 0
    sampling: int = 0
    bad: int = 0
    exact: int = 0
    excused_accept: int = 0
    excused_cdf: int = 0
    failures: list = field(default_factory=list)

    @property
    def excused(self) -> int:
        return self.excused_accept + self.excused_cdf

    def summary(self) -> str:
        return (f"requests={self.requests} greedy={self.greedy} sampling={self.sampling} "
                f"bad={self.bad} exact={self.exact} excused_accept={self.excused_accept} "
                f"excused_cdf={self.excused_cdf} failures={len(self.failures)}")


def compare_tree(inp: dict, ids, nacc, last, dbg, ref: dict, req_index=None) -> TreeReport:
    T = inp["temperature"]
    B = T.shape[0]
    rep = TreeReport(requests=B)
    probe = []
    for b in range(B):
        ao = int(ref["out_num_accepted"][b])
        if ao == -1:
            rep.bad += 1
            if nacc[b] != -1 or (ids[b] != -1).any():
                rep.failures.append((b, "bad request not rejected"))
            continue
        same = (nacc[b] == ao and last[b] == ref["out_last_node"][b]
                and np.array_equal(ids[b], ref["out_ids"][b]))
        if T[b] == 0:
            rep.greedy += 1
            if same:
                rep.exact += 1
            else:
                rep.failures.append((b, "greedy mismatch", ref["out_ids"][b].tolist(),
                                     ids[b].tolist()))
            continue
        rep.sampling += 1
        if same:
            rep.exact += 1
            continue
        # the first child the two walks decided differently
        nd = ref["node_diag"][b]
        div = None
        for c in range(1, ids.shape[1]):
            ro, rg = nd[c, oracle.R_ACCEPT], dbg[b, c, 3]
            if ro >= 0 and rg >= 0 and int(ro) != int(rg):
                div = c
                break
        if div is not None:
            u, r, q = nd[div, oracle.R_U], nd[div, oracle.R_PX], nd[div, oracle.R_QX]
            ratio = r / q if q > 0 else np.inf
            if abs(u - ratio) < TIE:
                rep.excused_accept += 1
            else:
                rep.failures.append((b, "tree accept mismatch", div, u, ratio))
            continue
        if nacc[b] != ao or last[b] != ref["out_last_node"][b] or \
                not np.array_equal(ids[b, :ao], ref["out_ids"][b, :ao]):
            rep.failures.append((b, "path mismatch", ref["out_ids"][b].tolist(), ids[b].tolist()))
            continue
        probe.append(b)
    if probe:
        sel = np.array(probe)
        sub = {k: (v[sel] if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
        gidx = sel if req_index is None else req_index[sel]
        pr = np.array([ids[b, nacc[b]] for b in sel], np.int32)
        r2 = oracle.tree_verify(**sub, req_index=gidx, probe=pr)
        for i, b in enumerate(sel):
            d = r2["req_diag"][i]
            u2, lo, hi = d[oracle.Q_UEMIT], d[oracle.Q_PLO], d[oracle.Q_PHI]
            if hi > lo and lo - TIE < u2 <= hi + TIE:
                rep.excused_cdf += 1
            else:
                rep.failures.append((int(b), "emitted token mismatch", float(u2), float(lo),
                                     float(hi)))
    return rep
