"""The seeded synthetic MoE-layer workloads (shapes, routers, seeds).

Shapes follow the model families the pages name: a tiny layer, an
OLMoE-shaped layer, a Mixtral-8x7B-shaped layer and GLM-5.2-style decode and
prefill layers (colibrì engine teardown, text-matrix.pages.dev, "System map":
256 routed experts of about 19 MB int4 each, 8 active per token, plus a
shared expert).  No dataset and no trained weight is involved.
"""
from dataclasses import dataclass, field
from typing import Tuple

ROUTER_SOFTMAX = 0
ROUTER_SIGMOID = 1
ROUTER_SOFTMAX_RAW = 2      # softmax top-k without renormalisation
X_F32 = 0
X_BF16 = 1


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    E: int
    k: int
    I: int
    n_shared: int
    I_shared: int
    router_mode: int
    rsf: float
    x_dtype: int
    tokens: Tuple[int, ...]
    seed: int
    layers: int = 1
    bias: str = "none"          # "none" | "normal" | "zipf"
    bias_sigma: float = 0.0
    zipf_s: float = 0.0
    router_sigma: float = 0.02
    n_group: int = 0            # > 1: grouped noaux_tc (sigmoid router)
    topk_group: int = 0
    top_p: float = 0.0          # adaptive expert top-p; 0: off
    scale_lo: float = 0.005
    scale_hi: float = 0.02
    notes: str = field(default="", compare=False)

    @property
    def bytes_per_expert(self):
        """Packed int4 + f32 gs64 scales of W1, W3 and W2 (0.5625 B per weight)."""
        return 3 * self.H * self.I * 9 // 16

    @property
    def bytes_shared(self):
        return 3 * self.H * self.I_shared * 9 // 16 if self.n_shared else 0


TINY = Workload("tiny", H=512, E=8, k=2, I=1024, n_shared=0, I_shared=0,
                router_mode=ROUTER_SOFTMAX, rsf=1.0, x_dtype=X_F32, tokens=(16,), seed=0,
                notes="tiny softmax layer, x f32")
OLMOE = Workload("olmoe", H=2048, E=64, k=8, I=1024, n_shared=0, I_shared=0,
                 router_mode=ROUTER_SOFTMAX, rsf=1.0, x_dtype=X_BF16, tokens=(1, 64), seed=2,
                 bias="zipf", zipf_s=1.0,
                 notes="OLMoE-shaped; seeded per-expert logit offset gives Zipf(1.0) popularity")
MIXTRAL = Workload("mixtral", H=4096, E=8, k=2, I=14336, n_shared=0, I_shared=0,
                   router_mode=ROUTER_SOFTMAX, rsf=1.0, x_dtype=X_BF16, tokens=(1, 4, 512),
                   seed=3, notes="Mixtral-8x7B-shaped, uniform routing")
GLM_DECODE = Workload("glm_decode", H=6144, E=256, k=8, I=2048, n_shared=1, I_shared=2048,
                      router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_BF16, tokens=(1, 2, 4),
                      seed=4, layers=8, bias="normal", bias_sigma=0.1,
                      notes="GLM-5.2-style decode stack of 8 layers with residual")
GLM_PREFILL = Workload("glm_prefill", H=6144, E=256, k=8, I=2048, n_shared=1, I_shared=2048,
                       router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_BF16, tokens=(4096,),
                       seed=5, bias="zipf", zipf_s=1.2,
                       notes="GLM-5.2-style prefill layer, Zipf(1.2) expert loads")

# A reduced GLM-shaped prefill layer (32 experts, uniform-ish routing) that
# holds ~2.5 GB on the device: the case the detailed kernel profiles capture.
GLM_PREFILL_SMALL = Workload("glm_prefill_small", H=6144, E=32, k=8, I=2048, n_shared=1,
                             I_shared=2048, router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_BF16,
                             tokens=(2048,), seed=6, bias="normal", bias_sigma=0.1,
                             notes="GLM-shaped layer with 32 experts, for kernel profiles")

# Router variants (the same shapes, other selection rules).
TINY_GROUPED = Workload("tiny_grouped", H=512, E=8, k=2, I=1024, n_shared=0, I_shared=0,
                        router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_F32, tokens=(16,),
                        seed=10, bias="normal", bias_sigma=0.1, n_group=4, topk_group=2,
                        notes="tiny sigmoid layer, 4 groups of 2 experts, 2 groups kept")
TINY_TOPP = Workload("tiny_topp", H=512, E=8, k=4, I=1024, n_shared=0, I_shared=0,
                     router_mode=ROUTER_SOFTMAX, rsf=1.0, x_dtype=X_F32, tokens=(16,), seed=11,
                     top_p=0.6, notes="tiny softmax layer with adaptive top-p 0.6")
OLMOE_RAW = Workload("olmoe_raw", H=2048, E=64, k=8, I=1024, n_shared=0, I_shared=0,
                     router_mode=ROUTER_SOFTMAX_RAW, rsf=1.0, x_dtype=X_BF16, tokens=(1, 64),
                     seed=12, bias="normal", bias_sigma=0.5,
                     notes="OLMoE-shaped, softmax top-k weights left unrenormalised")
GLM_GROUPED = Workload("glm_grouped", H=6144, E=256, k=8, I=2048, n_shared=1, I_shared=2048,
                       router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_BF16, tokens=(1, 4, 512),
                       seed=13, bias="normal", bias_sigma=0.1, n_group=8, topk_group=4,
                       notes="GLM-shaped layer, grouped noaux_tc: 8 groups of 32, 4 kept")
GLM_TOPP = Workload("glm_topp", H=6144, E=256, k=8, I=2048, n_shared=1, I_shared=2048,
                    router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_BF16, tokens=(1, 4, 512),
                    seed=14, bias="normal", bias_sigma=0.1, top_p=0.7,
                    notes="GLM-shaped layer with adaptive expert top-p 0.7")

# Many fine-grained experts with a wide top-k (the routing limits: 1024
# experts, 16 slots, so a token has more than 256 segment candidates).
WIDE = Workload("wide", H=512, E=1024, k=16, I=1024, n_shared=1, I_shared=1024,
                router_mode=ROUTER_SIGMOID, rsf=2.5, x_dtype=X_F32, tokens=(1, 8, 24), seed=15,
                bias="normal", bias_sigma=0.1,
                notes="1024 small experts, top-16, sigmoid with bias, shared expert")

ALL = (TINY, OLMOE, MIXTRAL, GLM_DECODE, GLM_PREFILL, GLM_PREFILL_SMALL, TINY_GROUPED,
       TINY_TOPP, OLMOE_RAW, GLM_GROUPED, GLM_TOPP, WIDE)
BY_NAME = {w.name: w for w in ALL}
