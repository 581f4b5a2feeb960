"""Seeded synthetic inputs for the bounded-tree speculative decoding path.

This module only draws random numbers in the shapes of the pages' workloads;
it holds none of the method's arithmetic.  Both the CUDA path (tests,
benchmark) and the float64 oracle consume what it returns.

Workloads (a Qwen-size vocabulary V = 151936, drafter block L = 16, bf16):

* tiny:     drafter logits [L=4, V=32] fp32 ~ N(0, 2^2); target row of a node
            at depth d = drafter row min(d, L-1) + N(0, 1).
* zipf:     drafter row j: z_j(a) = -1.1 * ln(1 + sigma_j(a)) + G_{j,a}, with
            sigma_j a seeded permutation of 0..V-1 and G ~ Gumbel(0, 1)
            (a Gumbel-perturbed Zipf(s = 1.1) field at temperature 1);
            target row of a node at depth d = drafter row min(d, L-1)
            + N(0, 1.5^2); both rounded to bf16.
* mixture:  per tree two latent futures F1, F2, each a zipf field with its own
            permutations; drafter mode k = F_{k mod 2} + N(0, 1); the target
            follows one future chosen uniformly per tree, at row min(d, L-1),
            + N(0, 1.5^2).

The pages measure on public benchmarks and trained models (dialogue, code and
maths prompts on Qwen3 targets); none of those are used here, and these seeded
fields stand in for them.
"""
from __future__ import annotations

import torch

V_QWEN = 151936
BASE_SEED = 20261202


def seed_for(config: int, tree: int = 0) -> int:
    """Seed of tree `tree` in workload `config` (base + 1000 * config + tree)."""
    return BASE_SEED + 1000 * config + tree


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def tiny_drafter(seed: int, L: int = 4, V: int = 32) -> torch.Tensor:
    """[L, V] float32 ~ N(0, 2^2), on the CPU."""
    g = _gen(seed, "cpu")
    return 2.0 * torch.randn(L, V, generator=g, dtype=torch.float32)


def tiny_target(drafter: torch.Tensor, depth, seed: int) -> torch.Tensor:
    """[n, V] float32: drafter row min(depth, L-1) + N(0, 1) per node."""
    g = _gen(seed, "cpu")
    L, V = drafter.shape
    d = torch.as_tensor(depth, dtype=torch.long).clamp(0, L - 1)
    return drafter[d] + torch.randn(d.numel(), V, generator=g, dtype=torch.float32)


def zipf_field(rows: int, V: int, g: torch.Generator, device, s: float = 1.1) -> torch.Tensor:
    """[rows, V] float32 Gumbel-perturbed Zipf(s) logits with one random
    permutation of the ranks per row."""
    perm = torch.argsort(torch.rand(rows, V, generator=g, device=device), dim=1)
    base = -s * torch.log1p(perm.to(torch.float32))
    u = torch.rand(rows, V, generator=g, device=device).clamp_(min=1e-12, max=1.0 - 1e-7)
    return base - torch.log(-torch.log(u))


def zipf_drafter(n_trees: int, L: int, V: int, seed: int, device="cpu",
                 dtype=torch.bfloat16, seeds=None) -> torch.Tensor:
    """[n_trees, 1, L, V] drafter logits, tree t seeded with seeds[t]
    (default seed + t)."""
    out = torch.empty(n_trees, 1, L, V, dtype=dtype, device=device)
    for t in range(n_trees):
        g = _gen(seeds[t] if seeds is not None else seed + t, device)
        out[t, 0] = zipf_field(L, V, g, device).to(dtype)
    return out


def target_from_rows(rows: torch.Tensor, depth, sigma: float, seed: int,
                     dtype=torch.bfloat16, out: torch.Tensor | None = None) -> torch.Tensor:
    """[n, V] target logits: rows[min(depth, L-1)] + N(0, sigma^2), per node.

    rows: [L, V] logits (any float dtype) on the device the noise is drawn on.
    """
    device = rows.device
    g = _gen(seed, device)
    L, V = rows.shape
    d = torch.as_tensor(depth, dtype=torch.long, device=device).clamp(0, L - 1)
    n = d.numel()
    res = out if out is not None else torch.empty(n, V, dtype=dtype, device=device)
    step = max(1, (1 << 26) // max(V, 1))
    for i in range(0, n, step):
        j = min(n, i + step)
        noise = torch.randn(j - i, V, generator=g, device=device, dtype=torch.float32)
        res[i:j] = (rows[d[i:j]].to(torch.float32) + sigma * noise).to(res.dtype)
    return res


def mixture_drafter(n_trees: int, K: int, L: int, V: int, seed: int, device="cpu",
                    dtype=torch.bfloat16):
    """[n_trees, K, L, V] drafter logits from two latent futures per tree, and
    the [n_trees, 2, L, V] future fields plus the future the target follows."""
    drafter = torch.empty(n_trees, K, L, V, dtype=dtype, device=device)
    futures = torch.empty(n_trees, 2, L, V, dtype=torch.float32, device=device)
    choice = []
    for t in range(n_trees):
        g = _gen(seed + t, device)
        for f in range(2):
            futures[t, f] = zipf_field(L, V, g, device)
        for k in range(K):
            noise = torch.randn(L, V, generator=g, device=device, dtype=torch.float32)
            drafter[t, k] = (futures[t, k % 2] + noise).to(dtype)
        choice.append(int(torch.randint(0, 2, (1,), generator=g, device=device).item()))
    return drafter, futures, choice


def uniform_depths(B: int, L: int) -> list:
    """A nominal depth profile (used only when no tree is at hand): the root at
    depth 0 and the B other nodes spread evenly over depths 1..L."""
    return [0] + [1 + (i * L) // max(B, 1) for i in range(B)]
