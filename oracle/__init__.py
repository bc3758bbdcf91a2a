"""CPU oracle for the tensor-parallel transformer-block math.  TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct restatement, in numpy float64,
of what the three source pages say the method computes:

* "v4:Tensor Parallel 与 Sequence Parallel" (the TP/SP page): column- and
  row-parallel linears, the f/g operators, the TP MLP (GeLU and SwiGLU),
  bias placement, sequence-parallel token slabs, vocab-parallel cross-entropy.
* "TP 的 communication:一层几次?每次多少数据?" (the TP-communication page):
  all-reduce = reduce-scatter + all-gather, the per-rank traffic and the
  FLOPs-per-byte closed forms.
* "Generalized Tensor Parallelism(GTP)是什么?" (the GTP page): GTP_remat
  weight shards, the gather/prefetch chain, the weight-gradient
  reduce-scatter and its one-layer-deferred finalize.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The CUDA library
never imports, links or calls anything here, and nothing here calls the CUDA
library: the two share no code.  Inputs arrive as numpy arrays (the bf16
values widened exactly to float64); outputs are float64 unless a function
says it mirrors a bf16/fp32 rounding sequence.

Parity status: every public function is pinned by a ``-m "not gpu"`` test
against the pages' worked examples, closed forms, brute force or finite
differences; see ``tests/test_oracle_*.py``.
"""
from . import accounting, attention, collectives, embedding, gtp, numerics, tp_mlp, vocab_ce  # noqa: F401
