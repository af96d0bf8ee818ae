"""Workload table for the routed ReLU^2 MoE layer (shapes only, no arithmetic).

Five workloads, named by what they are:

* ``tiny_fp32``      hidden 256, 8 experts, top-2, one group, FP32 throughout.
* ``nano_decode``    hidden 2688, 128 experts, top-6, one group, BF16, T in {1,4,16,64}.
* ``nano_prefill``   the same layer at T in {2048, 8192, 32768}, with expert
                     popularity bent to Zipf(1.1) through the selection bias.
* ``super_latent``   hidden 4096, latent 1024, 512 experts, top-22, 8 groups
                     keeping 4, BF16, T in {1, 16, 256, 4096}.
* ``super_nvfp4``    the latent layer with NVFP4 routed experts, Zipf(1.1)
                     popularity, T in {1, 64, 8192}.

The Nano and Super widths are the ones the NemotronH pages name: 128 routed
experts plus one shared expert with six selected per token ("Nemotron Is Not One
Circuit", section "One Family, Multiple Circuits"); Super's 512 experts, top-22,
1024-wide latent and 2688x1024 expert matrices ("Nemotron-3.5-Super 120B on an
8 GB GPU", section "The only number that matters: bytes per token").

A ``router_only_grouped`` case (128 experts, top-6, eight groups keeping three)
reproduces the router parity case of "Nemotron Is Not One Circuit", section
"What CKE Has Actually Established".
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Tuple

# dtype codes; the same numbers are used by the C ABI (moe_dtype_t)
F32 = 0
BF16 = 1
NVFP4 = 2


@dataclass(frozen=True)
class MoEShape:
    name: str
    d_model: int
    d_latent: int          # 0 = experts act on the hidden width
    n_experts: int
    top_k: int
    n_group: int
    topk_group: int
    d_expert: int          # expert intermediate width I
    d_shared: int          # shared expert intermediate width S (0 = none)
    routed_scaling_factor: float
    norm_topk_prob: int = 1
    act_dtype: int = BF16
    expert_dtype: int = BF16
    zipf_s: float = 0.0    # 0 = no popularity skew
    relu_sparsity: float = 0.0   # 0 = plain random layer; else the fraction of expert neurons ReLU^2 zeroes
    weight_seed: int = 0   # workloads that are "the same layer" share this
    tokens: Tuple[int, ...] = field(default_factory=tuple)

    @property
    def d_e(self) -> int:
        """Width the routed experts act on."""
        return self.d_latent if self.d_latent else self.d_model

    @property
    def latent(self) -> bool:
        return self.d_latent > 0


TINY_FP32 = MoEShape("tiny_fp32", 256, 0, 8, 2, 1, 1, 128, 256, 2.5,
                     act_dtype=F32, expert_dtype=F32, weight_seed=0, tokens=(16,))
NANO_DECODE = MoEShape("nano_decode", 2688, 0, 128, 6, 1, 1, 1856, 3712, 2.5,
                       weight_seed=1, tokens=(1, 4, 16, 64))
NANO_PREFILL = replace(NANO_DECODE, name="nano_prefill", zipf_s=1.1,
                       tokens=(2048, 8192, 32768))
SUPER_LATENT = MoEShape("super_latent", 4096, 1024, 512, 22, 8, 4, 2688, 5376, 5.0,
                        weight_seed=3, tokens=(1, 16, 256, 4096))
SUPER_NVFP4 = replace(SUPER_LATENT, name="super_nvfp4", expert_dtype=NVFP4,
                      zipf_s=1.1, tokens=(1, 64, 8192))
# decode with the ReLU^2 sparsity of a trained layer (page "Nemotron-3.5-Super
# 120B on an 8 GB GPU", section "The engine, step by step", item 4: 92.5 % of
# an expert's neurons are zero for a token); inputs for the ReLU^2-sparse down
NANO_DECODE_SPARSE = replace(NANO_DECODE, name="nano_decode_relu_sparse", relu_sparsity=0.925,
                             tokens=(1, 2, 4, 16, 64))
SUPER_NVFP4_SPARSE = replace(SUPER_NVFP4, name="super_nvfp4_relu_sparse", relu_sparsity=0.925, zipf_s=0.0,
                             tokens=(1, 2, 4))
ROUTER_ONLY_GROUPED = MoEShape("router_only_grouped", 2688, 0, 128, 6, 8, 3, 1856, 3712, 2.5,
                               weight_seed=5, tokens=(64,))

WORKLOADS = {s.name: s for s in (TINY_FP32, NANO_DECODE, NANO_PREFILL,
                                  SUPER_LATENT, SUPER_NVFP4, ROUTER_ONLY_GROUPED,
                                  NANO_DECODE_SPARSE, SUPER_NVFP4_SPARSE)}


def scaled(shape: MoEShape, **kw) -> MoEShape:
    """A smaller copy of a workload (same structure) for fast tests."""
    return replace(shape, **kw)
