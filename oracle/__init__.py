"""CPU oracle of the pooled-wave MoE layer forward -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy statement of what the layer computes, written
from the pages' description of the Marin 535B-A23B MoE branch.  Only the test
suite, the package's smoke check and the benchmark's CPU-baseline leg may
import it; the CUDA library never calls it and shares no code with it.

Sources (cited by title and section):

* [LJ-HK] lamjinlab, "Marin 開始公開訓練 535B 參數 MoE 模型" (zh-HK),
  section 二 "稀疏模型的組織方式" (layer structure, latent projection,
  fixed pooled-wave all-to-all, the two capacity factors, drop-and-count) and
  section 四 (shared experts as a dense backbone when routed slots drop).
* [LJ-JA] lamjinlab, "Marin、535BパラメータMoEモデルのオープントレーニングを開始"
  (ja), section 二 "スパースモデルの構成": the same statements.
* [CSDN] devpress.csdn.net, "从玩具到前沿:训练一个真正的大模型,到底难在哪里",
  section 四 (Grug MoE) and appendix A.2 (quantile-balancing bias added to the
  router logits).

Every function in ``moe_layer`` is pinned by the ``-m "not gpu"`` tests
(brute force, closed forms, invariants, library special cases); none is
"parity unpinned".
"""
from .moe_layer import *  # noqa: F401,F403
