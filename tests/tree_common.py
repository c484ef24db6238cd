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

import oracle
from speculative_decoding_verification_51_gb300.workloads import (  # noqa: F401
    TreeWorkload, make_tree_workload, random_parents)

TIE = 1e-6


@dataclass
class TreeReport:
    requests: int = 0
    rows: int = 0  # node rows of the batch (B x N)
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
    rep = TreeReport(requests=B, rows=int(np.asarray(inp["tree_tokens"]).size))
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
