"""The five synthetic MoGE workloads (shapes, dtypes, input recipe).

K' (experts per group) is explicit in every workload; K = M * K'.  The
routing-only workload is also run at K' = 1.  The prefill and decode layers
share one layer shape (d=4096, N=64 in 8 groups, K'=2, I=1408); the stress
layer borrows the Pangu Ultra MoE dimensions (d=7680, N=256, I=2048) with
MoGE routing imposed on them.  The two "pangu_k1" layers take Pangu Pro MoE's
own dimensions (hidden 5120, 64 routed experts in 8 groups, top-1 per group,
i.e. K = 8; 4 shared experts are added where they are measured) with an expert
intermediate size of 1344, which the pages do not give: 48 layers x 68 experts
x 3*5120*1344 weights is about 67 B parameters, consistent with the 72 B total
they print once attention and embeddings are counted.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

DEFAULT_SEED = 20250527


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    N: int
    M: int
    kpg: int          # K' = experts selected per group
    I: int
    dtype: str        # "f32" or "bf16" for activations and weights
    skew: bool        # add the seeded popularity bias b_e = 1.5 ln(1/rank_e)
    routing_only: bool = False

    @property
    def G(self) -> int:
        return self.N // self.M

    @property
    def K(self) -> int:
        return self.M * self.kpg

    @property
    def P(self) -> int:
        return self.T * self.K

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=256, N=16, M=4, kpg=1, I=128,
                          dtype="f32", skew=False),
    "routing_16k": Workload("routing_16k", T=16384, d=0, N=64, M=8, kpg=2, I=0,
                            dtype="f32", skew=True, routing_only=True),
    "decode_t32": Workload("decode_t32", T=32, d=4096, N=64, M=8, kpg=2, I=1408,
                           dtype="bf16", skew=True),
    "prefill_t8192": Workload("prefill_t8192", T=8192, d=4096, N=64, M=8, kpg=2, I=1408,
                              dtype="bf16", skew=True),
    "stress_n256": Workload("stress_n256", T=4096, d=7680, N=256, M=8, kpg=1, I=2048,
                            dtype="bf16", skew=True),
    "pangu_k1_t32": Workload("pangu_k1_t32", T=32, d=5120, N=64, M=8, kpg=1, I=1344,
                             dtype="bf16", skew=True),
    "pangu_k1_t8192": Workload("pangu_k1_t8192", T=8192, d=5120, N=64, M=8, kpg=1, I=1344,
                               dtype="bf16", skew=True),
}
