"""Layer dimensions shared by the binding, the input generator and the tests.

Plain data only.  The fields follow the MoE layer arguments the vLLM
specialized-decode page (vllm.models.glm5next.nvidia.specialized_decode.runtime
.decode, LayerStages._build_mega) hands to its expert kernels:
num_experts_per_tok (top_k), swiglu_limit, routed_scaling_factor and the e8m0
scale switch, plus the hidden / intermediate sizes of the weights and the norm
epsilon of the layer boundary.
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerDims:
    hidden: int  # H
    inter: int  # I, routed expert intermediate size
    shared_inter: int  # I_s, shared expert intermediate size (0: no shared expert)
    num_experts: int  # E
    top_k: int  # k
    routed_scaling: float = 2.5
    swiglu_limit: float = 7.0
    rms_eps: float = 1e-6
    e8m0: bool = False

    def with_(self, **kw) -> "LayerDims":
        return replace(self, **kw)


# Tiny MoE decode layer: H=512, 16 routed experts, top-4, I = I_s = 256.
TINY = LayerDims(hidden=512, inter=256, shared_inter=256, num_experts=16, top_k=4)
# DeepSeek-V3-shaped decode layer: H=7168, 256 routed experts, top-8, I = I_s = 2048.
DSV3 = LayerDims(hidden=7168, inter=2048, shared_inter=2048, num_experts=256, top_k=8)
# Dense layers (num_experts = 0): the MLP in the shared-expert slot, no router
# ([decode page] LayerStages._build_dense runs dense MLPs as GEMVs).
TINY_DENSE = LayerDims(hidden=512, inter=0, shared_inter=768, num_experts=0, top_k=0)
# DeepSeek-V3's dense layers: H = 7168, intermediate 18432.
DSV3_DENSE = LayerDims(hidden=7168, inter=0, shared_inter=18432, num_experts=0, top_k=0)
