"""CPU oracle of the Megatron column/row-parallel transformer block.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import or run anything in this package. The
CUDA library never calls it, links it or falls back to it; it shares no code
with the CUDA path (the seeded input generator in ``synth.py`` is the only
module both sides use, and it holds none of the block's arithmetic).

Everything here is plain numpy in float64 on inputs already rounded to their
storage type, with no intermediate rounding. Library matmuls serve as steps;
there is no blocking, fusion or reordering beyond what each function's
docstring states.

Sources, cited by page title and section:

* "feat: multi-GPU tensor-parallel runtime with per-rank device placement and
  cross-GPU collectives" (the mlxcel TP-runtime issue): sections Problem and
  Design / Forward execution (replicated residual stream, reduction after
  o_proj and after down_proj) and Collective backend abstraction
  (copy-and-reduce: gather the partials, sum, broadcast).
* "Gather tensor-parallel sharded parameters on read in a trace" (the nnsight
  gather-on-read PR): section Change (shard-dim rule, replicated tensors,
  vocab padding dropped to org_vocab_size, fused rows grouped by rank) and
  section Verification (the checks used: row-parallel gather equal to the
  tp=1 tensor, fused weights equal as a row multiset, lm_head row vocab-5).
* "Multi-GPU & Multi-Node" (the TensorSharp docs): section How tensor
  parallelism works (steps 1-3 and the replicated norms paragraph), section
  Supported architectures (expert slicing, and expert parallelism with whole
  experts per rank, both with a replicated router) and section Requirements &
  constraints (divisibility).

The per-op formulas (RMSNorm, rotate-half RoPE, GQA head grouping, SwiGLU) are
not written out on the pages; the workload descriptions name them and the
oracle uses their textbook definitions.

Parity status: every function in ``block.py`` is pinned by ``-m "not gpu"``
tests against closed forms, library routines, brute force on tiny inputs or
the pages' stated invariants. The end-to-end block has no worked numeric
example on the pages, so beyond those pins its absolute values rest on the
agreement of independent formulations (see ``tests/test_oracle_pins.py``).
"""
from .block import *  # noqa: F401,F403
