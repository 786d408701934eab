"""Plain, slow, fp64 CPU oracle for FlashAttention-2 exact attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
package: only the test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA library (``exact_attention_64_gb300``), and the CUDA
library never calls it.

Modules
-------
attention  -- softmax(scale*Q K^T + causal mask) V, its logsumexp, and the
              naive chain-rule backward (the definition FlashAttention-2 reaches
              exactly, up to rounding).
schedule   -- the integer work mapping the pages describe: the forward grid
              (num_m_block, batch, heads), the backward column workers, and the
              causal rule that drops fully masked key/query tiles.

Parity pins: every function here is pinned by ``tests/test_oracle*.py`` against
closed forms, brute force, finite differences, invariants, a library special
case and the pages' own worked grid example. No function is "parity unpinned".
"""

from .attention import forward, backward, lse_brute_force, combine_partials  # noqa: F401
from .schedule import (  # noqa: F401
    fwd_grid,
    fwd_work_order,
    fwd_kv_tile_range,
    bwd_grid,
    bwd_q_tile_range,
)
