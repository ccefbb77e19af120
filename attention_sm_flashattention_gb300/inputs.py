"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests
and the benchmark.

This module holds no attention arithmetic: it only names the workloads and
draws their tensors.  Recipe: a CPU ``torch.Generator`` seeded with the
workload's seed draws ``q``, ``k``, ``v``, ``do`` in that order, each as
standard-normal float32 of shape ``[Z, H, N, D]`` (k and v ``[Z, Hkv, Nk, D]``
for grouped heads or unequal lengths), then rounds them to fp16
(round-to-nearest-even), or to bf16 for the bf16 path.  ``scale = 1/sqrt(D)`` passed as a float32.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    Z: int
    H: int
    N: int
    D: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def heads(self) -> int:
        return self.Z * self.H

    def describe(self) -> str:
        kind = "causal" if self.causal else "non-causal"
        return f"Z{self.Z} H{self.H} N{self.N} D{self.D} {kind}"


# The five benchmark shapes (the D256 one in both masks).  Seeds: 1000 + the
# shape's index, +10 for the causal variant of the D256 shape.
WORKLOADS = {
    "z1h2n128d64": Workload("z1h2n128d64", 1, 2, 128, 64, False, 1000),
    "z4h8n1024d64": Workload("z4h8n1024d64", 4, 8, 1024, 64, False, 1001),
    "z128h8n1024d128": Workload("z128h8n1024d128", 128, 8, 1024, 128, False, 1002),
    "z128h8n1024d128c": Workload("z128h8n1024d128c", 128, 8, 1024, 128, True, 1003),
    "z128h8n1024d256": Workload("z128h8n1024d256", 128, 8, 1024, 256, False, 1004),
    "z128h8n1024d256c": Workload("z128h8n1024d256c", 128, 8, 1024, 256, True, 1014),
}


def make_inputs(Z: int, H: int, N: int, D: int, seed: int, device="cpu", dtype=torch.float16,
                Hkv: int | None = None, Nk: int | None = None):
    """Draw ``(q, k, v, do)`` from ``seed``, rounded to ``dtype`` (fp16 by
    default, or bf16; the same draw either way).  q and do are
    ``[Z, H, N, D]``; k and v are ``[Z, Hkv, Nk, D]`` (``Hkv = H``, ``Nk = N``
    unless given: grouped K/V heads and unequal query / key lengths).

    The draw always happens on the CPU generator so that every device sees
    bit-identical tensors; ``device`` only says where the result is moved.
    """
    Hkv = H if Hkv is None else Hkv
    Nk = N if Nk is None else Nk
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    shapes = ((Z, H, N, D), (Z, Hkv, Nk, D), (Z, Hkv, Nk, D), (Z, H, N, D))
    out = []
    for shape in shapes:
        t = torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)
        out.append(t if device == "cpu" else t.to(device))
    return tuple(out)


def workload_inputs(w: Workload, device="cpu"):
    return make_inputs(w.Z, w.H, w.N, w.D, w.seed, device=device)


def make_paged_inputs(B: int, H: int, Hkv: int, Nq: int, context_lens, D: int, page_size: int, seed: int,
                      spare_pages: int = 3, device="cpu", dtype=torch.float16):
    """Draw a paged-cache problem from ``seed``: ``(q, k_cache, v_cache,
    block_table, context_lens)``.

    q is ``[B, H, Nq, D]``; the caches are ``[num_pages, page_size, Hkv, D]``
    with every slot drawn (slots past a context length hold values too);
    sequence b owns ceil(context_lens[b] / page_size) pages, taken from a
    random permutation of all pages (``spare_pages`` more than needed), and
    its block-table row is padded with -1 to the longest sequence.  Draw
    order: q, k_cache, v_cache, page permutation.
    """
    lens = [int(x) for x in context_lens]
    need = [(n + page_size - 1) // page_size for n in lens]
    num_pages = sum(need) + spare_pages
    max_pages = max(need)
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    q = torch.randn((B, H, Nq, D), generator=g, dtype=torch.float32).to(dtype)
    kc = torch.randn((num_pages, page_size, Hkv, D), generator=g, dtype=torch.float32).to(dtype)
    vc = torch.randn((num_pages, page_size, Hkv, D), generator=g, dtype=torch.float32).to(dtype)
    perm = torch.randperm(num_pages, generator=g)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    pos = 0
    for b in range(B):
        table[b, :need[b]] = perm[pos:pos + need[b]].to(torch.int32)
        pos += need[b]
    cl = torch.tensor(lens, dtype=torch.int32)
    out = (q, kc, vc, table, cl)
    return out if device == "cpu" else tuple(t.to(device) for t in out)
