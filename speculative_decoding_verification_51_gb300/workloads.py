"""Seeded synthetic inputs for the speculative-sampling verifier.

This module only builds inputs: target logits, a simulated drafter's
distribution q and its sampled draft tokens, ragged draft counts and
temperatures.  It holds none of the verifier's arithmetic (no acceptance
test, no residual, no uniforms) and is shared by the CUDA path's tests, the
benchmark and the oracle's tests alike.

The five workloads (sizes, value distributions and structure) are the ones
the verifier is measured on:

  1. B=1,   K=4, V=1024,   f32  logits ~ N(0, 2^2); draft = target + N(0, 1);
     T = 1.
  2. B=8,   K=5, V=32000,  bf16 logits ~ N(0, 3^2) with +8 on one random
     token per row; draft = target + N(0, 1.5^2); odd requests greedy (T=0).
  3. B=64,  K=4, V=128256, bf16 Zipf(1.1) profile (logit of rank r is
     -1.1 ln r) placed by one random permutation per request, + N(0, 1) per
     element; draft = target + N(0, 1); T ~ U[0.5, 1.2].
  4. B=256, K=3, V=151936, bf16 as 3; num_draft ~ U{0..3}; 25% of requests
     greedy; draft noise sigma per request from {0.25, 1, 4}; T ~ U[0.5, 1.2].
  5. B=512, K=8, V=129280, bf16 as 3; draft = target + N(0, 0.5^2);
     num_draft ~ U{1..8}; T ~ U[0.3, 1.5]; B sweep {32, 128, 512} takes the
     leading requests.

The drafter: q = softmax(draft_logits / T_b) in float32 (T_b = 1 for greedy
requests, whose q the verifier never reads); sampling requests draw their
draft tokens from q, greedy requests take argmax(draft_logits).  Draft ids at
positions j >= num_draft[b] are set to -1: the verifier must never read them.
"""
from __future__ import annotations

import functools
from dataclasses import dataclass, field

import numpy as np
import torch

VERIFY_SEED = 0  # Philox seed of the verifier for every workload


@dataclass(frozen=True)
class WorkloadSpec:
    cid: int
    B: int
    K: int
    V: int
    dtype: str  # "f32" | "bf16"
    description: str


SPECS = {
    1: WorkloadSpec(1, 1, 4, 1024, "f32", "B=1 K=4 V=1024 f32 gaussian logits, T=1"),
    2: WorkloadSpec(2, 8, 5, 32000, "bf16", "B=8 K=5 V=32000 bf16 gaussian+boost, half greedy"),
    3: WorkloadSpec(3, 64, 4, 128256, "bf16", "B=64 K=4 V=128256 bf16 zipf, T~U[0.5,1.2]"),
    4: WorkloadSpec(4, 256, 3, 151936, "bf16",
                    "B=256 K=3 V=151936 bf16 zipf, ragged n~U{0..3}, 25% greedy"),
    5: WorkloadSpec(5, 512, 8, 129280, "bf16",
                    "B=512 K=8 V=129280 bf16 zipf, ragged n~U{1..8}, T~U[0.3,1.5]"),
}


@dataclass
class Workload:
    spec: WorkloadSpec
    target_logits: torch.Tensor  # [B, K+1, V] bf16 or f32
    draft_probs: torch.Tensor    # [B, K, V] f32
    draft_ids: torch.Tensor      # [B, K] int32 (-1 beyond num_draft)
    num_draft: torch.Tensor      # [B] int32
    temperature: torch.Tensor    # [B] f32 (0 = greedy)
    seed: int = VERIFY_SEED
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target_logits.shape[0]

    @property
    def K(self) -> int:
        return self.draft_probs.shape[1]

    @property
    def V(self) -> int:
        return self.target_logits.shape[2]

    def to(self, device) -> "Workload":
        return Workload(self.spec, self.target_logits.to(device), self.draft_probs.to(device),
                        self.draft_ids.to(device), self.num_draft.to(device),
                        self.temperature.to(device), self.seed, dict(self.meta))

    def subset(self, idx) -> "Workload":
        """Requests idx (a list or 1-D tensor of request indices)."""
        i = torch.as_tensor(idx, dtype=torch.long, device=self.target_logits.device)
        return Workload(self.spec, self.target_logits[i].contiguous(),
                        self.draft_probs[i].contiguous(), self.draft_ids[i].contiguous(),
                        self.num_draft[i].contiguous(), self.temperature[i].contiguous(),
                        self.seed, dict(self.meta))

    def leading(self, B: int) -> "Workload":
        return self.subset(list(range(B)))


def _zipf_logits(nb, K1, V, g):
    """-1.1 ln(rank) placed by one permutation per request, + N(0, 1) noise."""
    rank = torch.arange(1, V + 1, dtype=torch.float32)
    base = -1.1 * torch.log(rank)                                   # [V]
    perm = torch.argsort(torch.rand(nb, V, generator=g), dim=1)
    placed = torch.empty(nb, V, dtype=torch.float32)
    placed.scatter_(1, perm, base.expand(nb, V).contiguous())       # token perm[r] gets rank r
    noise = torch.randn(nb, K1, V, generator=g)
    return placed[:, None, :] + noise


# requests generated together (bounds the host memory of the largest workloads)
GEN_BLOCK = 32


def _draw(q: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """One token per row of q [R, V] (rows summing to about 1): the first
    token whose float64 running sum exceeds u * (row total), u ~ U[0, 1).
    A token of zero mass is never drawn."""
    cdf = torch.cumsum(q.to(torch.float64), dim=-1)
    u = torch.rand(q.shape[0], generator=g, dtype=torch.float64)
    t = (u * cdf[:, -1]).unsqueeze(1)
    x = torch.searchsorted(cdf, t, right=True).squeeze(1)
    return x.clamp_(max=q.shape[1] - 1)


def make_workload(cid: int, device="cpu", *, gen_seed: int | None = None, B: int | None = None,
                  K: int | None = None, V: int | None = None) -> Workload:
    """Build workload ``cid`` (1..5) from a seeded CPU generator, then copy it
    to ``device``: a named workload is one fixed set of inputs on every device.

    The per-request scalars (draft counts, temperatures, draft noise) are drawn
    first for the whole batch, then the rows request block by request block
    (GEN_BLOCK requests at a time), all from one generator stream.
    B, K, V override the sizes (for small parity cases of the same recipe).
    The host tensors of the last few workloads built are kept, so a repeated
    build only copies; every call returns tensors of its own.
    """
    spec = SPECS[cid]
    B = spec.B if B is None else B
    K = spec.K if K is None else K
    V = spec.V if V is None else V
    seed = 1000 + cid if gen_seed is None else gen_seed
    t = _generate(cid, seed, B, K, V)
    logits, probs, ids, num, temp = (x.to(device, copy=True) for x in t[:5])
    return Workload(spec, logits, probs, ids, num, temp, VERIFY_SEED,
                    {"gen_seed": seed, "draft_noise": t[5]})


@functools.lru_cache(maxsize=3)
def _generate(cid: int, seed: int, B: int, K: int, V: int):
    """Host tensors (logits, draft_probs, draft_ids, num_draft, temperature,
    draft noise list or None) of workload ``cid`` at these sizes."""
    spec = SPECS[cid]
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    K1 = K + 1
    f32 = torch.float32

    # ---- per-request scalars
    if cid == 1:
        draft_noise = torch.ones(B)
        num_draft = torch.full((B,), K, dtype=torch.int32)
        temp = torch.ones(B)
    elif cid == 2:
        draft_noise = torch.full((B,), 1.5)
        num_draft = torch.full((B,), K, dtype=torch.int32)
        temp = torch.ones(B)
        temp[1::2] = 0.0  # odd requests greedy
    elif cid == 3:
        draft_noise = torch.ones(B)
        num_draft = torch.full((B,), K, dtype=torch.int32)
        temp = 0.5 + 0.7 * torch.rand(B, generator=g)
    elif cid == 4:
        sig = torch.tensor([0.25, 1.0, 4.0])
        draft_noise = sig[torch.randint(0, 3, (B,), generator=g)]
        num_draft = torch.randint(0, K + 1, (B,), generator=g).to(torch.int32)
        temp = 0.5 + 0.7 * torch.rand(B, generator=g)
        greedy = torch.rand(B, generator=g) < 0.25
        temp = torch.where(greedy, torch.zeros_like(temp), temp)
    elif cid == 5:
        draft_noise = torch.full((B,), 0.5)
        num_draft = torch.randint(1, K + 1, (B,), generator=g).to(torch.int32)
        temp = 0.3 + 1.2 * torch.rand(B, generator=g)
    else:
        raise ValueError(f"unknown workload {cid}")
    temp = temp.to(f32)

    ldt = torch.bfloat16 if spec.dtype == "bf16" else f32
    logits = torch.empty((B, K1, V), dtype=ldt)
    draft_probs = torch.empty((B, K, V), dtype=f32)
    draft_ids = torch.full((B, K), -1, dtype=torch.int32)
    for b0 in range(0, B, GEN_BLOCK):
        b1 = min(B, b0 + GEN_BLOCK)
        nb = b1 - b0
        if cid == 1:
            target = 2.0 * torch.randn(nb, K1, V, generator=g)
        elif cid == 2:
            target = 3.0 * torch.randn(nb, K1, V, generator=g)
            boost = torch.randint(0, V, (nb, K1, 1), generator=g)
            target.scatter_add_(2, boost, torch.full((nb, K1, 1), 8.0))
        else:
            target = _zipf_logits(nb, K1, V, g)
        # the simulated drafter sees the first K rows of the target plus noise
        dlog = target[:, :K, :] + draft_noise[b0:b1, None, None] * torch.randn(
            nb, K, V, generator=g)
        tb = temp[b0:b1]
        t_draft = torch.where(tb > 0, tb, torch.ones_like(tb))
        q = torch.softmax(dlog / t_draft[:, None, None], dim=-1).to(f32).contiguous()
        if K > 0:
            sampled = _draw(q.reshape(nb * K, V), g).reshape(nb, K)
            greedy_ids = dlog.argmax(dim=-1)
            ids = torch.where((tb > 0)[:, None], sampled, greedy_ids).to(torch.int32)
            pos = torch.arange(K)[None, :]
            draft_ids[b0:b1] = torch.where(pos < num_draft[b0:b1, None].long(), ids,
                                           torch.full_like(ids, -1))
        logits[b0:b1] = target.to(ldt)
        draft_probs[b0:b1] = q
        del target, dlog, q

    return (logits, draft_probs, draft_ids.contiguous(), num_draft.contiguous(),
            temp.contiguous(), draft_noise.tolist() if B <= 16 else None)


def to_numpy(w: Workload) -> dict:
    """Host copies in the layout the oracle takes (bf16 as uint16 bit patterns)."""
    tl = w.target_logits.detach().cpu()
    if tl.dtype == torch.bfloat16:
        tl_np = tl.view(torch.int16).numpy().view("uint16")
    else:
        tl_np = tl.numpy()
    return {
        "target_logits": tl_np,
        "draft_probs": w.draft_probs.detach().cpu().numpy(),
        "draft_ids": w.draft_ids.detach().cpu().numpy(),
        "num_draft": w.num_draft.detach().cpu().numpy(),
        "temperature": w.temperature.detach().cpu().numpy(),
        "seed": w.seed,
    }


def valid_rows(num_draft: torch.Tensor) -> int:
    """Rows the verifier must read whole: sum_b (num_draft[b] + 1)."""
    return int((num_draft.long() + 1).sum().item())


def positions(num_draft: torch.Tensor) -> int:
    """Verified draft positions: sum_b num_draft[b]."""
    return int(num_draft.long().sum().item())


# ---------------------------------------------------------------- token trees
# Token-tree workloads (tries of drafts): node 0 is the accepted context, node
# c >= 1 a draft token under an earlier parent; row v of the logits scores the
# token after node v.  Target rows as above (Zipf profile + N(0, 1) noise);
# node c's draft distribution is a noisy copy of its parent's row.

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


# ---------------------------------------------------------------- hidden states
# Workloads of the fused logits producer: the target's last hidden states and
# an LM-head matrix instead of logits.  Both operands hold small integers
# (hidden in -3..3, LM head in -15..15 times a power of two s), so every
# float32 partial sum of the projection is a multiple of s below 2^24 s and
# exact in any order: the logits are the same on every path that sums in
# float32 or wider, before the one rounding to bf16.  s = 2^round(log2(2.5 /
# sqrt(320 H))) gives logits of standard deviation about 2.5.

@dataclass
class LmHeadWorkload:
    hidden: torch.Tensor       # [B, K+1, H] bf16
    lm_head: torch.Tensor      # [V, H] bf16
    draft_probs: torch.Tensor  # [B, K, V] f32
    draft_ids: torch.Tensor    # [B, K] int32 (-1 past num_draft)
    num_draft: torch.Tensor    # [B] int32
    temperature: torch.Tensor  # [B] f32 (0 = greedy)
    seed: int

    @property
    def shape(self):
        B, K1, H = self.hidden.shape
        return B, K1 - 1, self.lm_head.shape[0], H


def lmhead_scale(H: int) -> float:
    return 2.0 ** round(float(np.log2(2.5 / np.sqrt(320.0 * H))))


def make_lmhead_workload(B, K, V, H, *, seed=0, greedy_frac=0.25, ragged=True, noise=1.0,
                         device="cuda") -> LmHeadWorkload:
    g = torch.Generator(device="cpu").manual_seed(seed)
    K1 = K + 1
    s = lmhead_scale(H)
    hidden = torch.randint(-3, 4, (B, K1, H), generator=g, dtype=torch.int8)
    hidden = hidden.to(device).to(torch.bfloat16).contiguous()
    w = torch.randint(-15, 16, (V, H), generator=g, dtype=torch.int8)
    lm_head = (w.to(device).to(torch.float32) * s).to(torch.bfloat16).contiguous()
    num_draft = (torch.randint(0, K + 1, (B,), generator=g) if ragged
                 else torch.full((B,), K)).to(torch.int32)
    temp = 0.5 + 0.7 * torch.rand(B, generator=g)
    temp = torch.where(torch.rand(B, generator=g) < greedy_frac, torch.zeros_like(temp), temp)
    # the drafter sees the target's logits (exact float32 sums, bf16-rounded)
    # plus noise; logits are formed a few rows at a time to bound memory
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    probs = torch.empty((B, K, V), dtype=torch.float32, device=device)
    ids = torch.full((B, K), -1, dtype=torch.int32)
    gd = torch.Generator(device=device).manual_seed(seed + 1)
    wf = lm_head.float()
    for b0 in range(0, B, 16):
        b1 = min(B, b0 + 16)
        lg = (hidden[b0:b1, :K].float() @ wf.T).to(torch.bfloat16).float()  # [bb, K, V]
        dl = lg + noise * torch.randn(lg.shape, generator=gd, device=device)
        t = temp[b0:b1].to(device)
        tq = torch.where(t > 0, t, torch.ones_like(t))[:, None, None]
        q = torch.softmax(dl / tq, dim=-1)
        probs[b0:b1] = q
        samp = torch.multinomial(q.reshape(-1, V), 1, generator=gd).reshape(b1 - b0, K)
        greedy_ids = dl.argmax(-1)
        pick = torch.where((t > 0)[:, None], samp, greedy_ids).to(torch.int32).cpu()
        ids[b0:b1] = pick
    torch.backends.cuda.matmul.allow_tf32 = prev
    pos = torch.arange(K)[None, :]
    ids = torch.where(pos < num_draft[:, None].long(), ids, torch.full_like(ids, -1))
    return LmHeadWorkload(hidden, lm_head, probs.contiguous(), ids.to(device).contiguous(),
                          num_draft.to(device), temp.to(torch.float32).to(device), seed * 31 + 5)


def lmhead_to_numpy(w: LmHeadWorkload) -> dict:
    """Host copies: operands as bf16 bit patterns, the rest as the oracle takes them."""
    def bits(t):
        return t.detach().cpu().view(torch.int16).numpy().view("uint16")
    return {"hidden": bits(w.hidden), "lm_head": bits(w.lm_head),
            "draft_probs": w.draft_probs.cpu().numpy(), "draft_ids": w.draft_ids.cpu().numpy(),
            "num_draft": w.num_draft.cpu().numpy(), "temperature": w.temperature.cpu().numpy(),
            "seed": w.seed}
