"""Named MoE-layer workloads: shapes, routing mode and value distributions.

Each workload is a synthetic stand-in for one model's MoE FFN layer, at the shapes the
source pages give (Mixtral 8x7B, DeepSeek-V3, DeepSeek-V4-Flash, DeepSeek-V4-Pro) plus a
toy layer.  Only shapes and distributions live here; the layer's arithmetic does not.

Sources (page title, section):
  * Mixtral 8x7B: d=4096, d_ff=14336, E=8, top-2 -- "Mixture of Experts: router, token
    dispatch, grouped GEMM", section "Expert 里面是什么" (Mixtral table).
  * DeepSeek-V3: d=7168, d_ff=2048, E=256, top-8, 1 shared expert, node-limited routing
    over 8 groups keeping 4 -- "MoE compute and communication", sections 二.4 and 五.3;
    "DeepSeek-V4 MoE", section "V3 的节点路由约束".
  * DeepSeek-V4-Flash / Pro: E=256/384, d_ff=2048/3072, top-6, 1 shared expert,
    sqrt(softplus) affinity, hash routing in the first layers -- "DeepSeek-V4 MoE",
    table "V4 MoE 基础配置" and eq. dsv4-moe-softplus; Pro hidden 7168 from eq.
    dsv4-moe-balance.  The V4-Flash hidden size (4096) is a chosen value.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

SCORE_SOFTMAX_TOPK = "softmax_topk"   # top-k on logits, softmax over the k selected
SCORE_SOFTMAX = "softmax"             # softmax over all E, top-k, renormalise
SCORE_SIGMOID = "sigmoid"
SCORE_SQRT_SOFTPLUS = "sqrt_softplus"
SCORES = (SCORE_SOFTMAX_TOPK, SCORE_SOFTMAX, SCORE_SIGMOID, SCORE_SQRT_SOFTPLUS)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens in the batch
    d: int                 # hidden size
    d_ff: int              # expert intermediate size (shared expert uses the same)
    E: int                 # routed experts
    k: int                 # experts per token
    n_shared: int          # 0 or 1
    score: str             # one of SCORES
    use_bias: bool = False         # per-expert selection bias ~ N(0, 0.01^2)
    n_groups: int = 0              # group-limited top-k (0 = off)
    topk_groups: int = 0
    group_topk: int = 0
    hash_vocab: int = 0            # > 0: HashTopK via tid2eid[vocab, k]
    zipf_s: float = 0.0            # > 0: per-expert additive logit offset -s*ln(1+rank)
    init: str = "std002"           # "std002": weights N(0, 0.02^2); "fan_in": N(0, 1/fan_in)

    @property
    def N(self) -> int:
        """Token-expert assignments T*k."""
        return self.T * self.k

    def with_T(self, T: int, name: Optional[str] = None) -> "Workload":
        return dataclasses.replace(self, T=T, name=name or f"{self.name.rsplit('_T', 1)[0]}_T{T}")


TOY = Workload("toy_T64", T=64, d=128, d_ff=64, E=8, k=2, n_shared=0,
               score=SCORE_SOFTMAX_TOPK, init="fan_in")
MIXTRAL_T16 = Workload("mixtral_T16", T=16, d=4096, d_ff=14336, E=8, k=2, n_shared=0,
                       score=SCORE_SOFTMAX)
MIXTRAL_T2048 = MIXTRAL_T16.with_T(2048, "mixtral_T2048")
V3_T4096 = Workload("v3_T4096", T=4096, d=7168, d_ff=2048, E=256, k=8, n_shared=1,
                    score=SCORE_SIGMOID, use_bias=True, n_groups=8, topk_groups=4,
                    group_topk=2, zipf_s=1.1)
V4FLASH_T64 = Workload("v4flash_T64", T=64, d=4096, d_ff=2048, E=256, k=6, n_shared=1,
                       score=SCORE_SQRT_SOFTPLUS, use_bias=True)
V4FLASH_T8192 = V4FLASH_T64.with_T(8192, "v4flash_T8192")
V4FLASH_T64_ZIPF = dataclasses.replace(V4FLASH_T64, name="v4flash_zipf_T64", zipf_s=1.1)
V4FLASH_T8192_ZIPF = dataclasses.replace(V4FLASH_T8192, name="v4flash_zipf_T8192", zipf_s=1.1)
V4PRO_HASH_T16384 = Workload("v4pro_hash_T16384", T=16384, d=7168, d_ff=3072, E=384, k=6,
                             n_shared=1, score=SCORE_SQRT_SOFTPLUS, hash_vocab=32768)
V4PRO_LEARNED_T16384 = Workload("v4pro_learned_T16384", T=16384, d=7168, d_ff=3072, E=384,
                                k=6, n_shared=1, score=SCORE_SQRT_SOFTPLUS, use_bias=True)

# Profiling stand-in: the V4-Flash layer's shapes with 32 experts and T=1024, i.e. the same
# 192 rows per expert as T=8192 over 256 experts, at 1.6 GB of expert weights (> L2).
V4FLASH_E32_T1024 = dataclasses.replace(V4FLASH_T8192, name="v4flash_E32_T1024", E=32, T=1024)

ALL = (TOY, MIXTRAL_T16, MIXTRAL_T2048, V3_T4096, V4FLASH_T64, V4FLASH_T8192,
       V4FLASH_T64_ZIPF, V4FLASH_T8192_ZIPF, V4PRO_HASH_T16384, V4PRO_LEARNED_T16384, V4FLASH_E32_T1024)
BY_NAME = {w.name: w for w in ALL}
