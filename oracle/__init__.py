"""CPU float64 oracle for the Dion3 optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may use it.  It shares no code with the CUDA path.

Functions and the passage each one follows are listed in ``dion3_oracle``.
Every function here is pinned by a ``-m "not gpu"`` test against something other
than itself (closed forms, SVD, brute force, the pages' FLOP figures); there is
no "parity unpinned" function in this package except the readings listed in
``dion3_oracle``'s header: the lr proportionality constant is taken as 1, and
the NorMuon per-neuron normalisation (``normuon_rows``, ``normuon_update``,
``dion3_step_normuon``) follows the NorMuon method, not the pages, which never
define it (PARITY UNPINNED as to the pages; pinned to its stated definition).
"""
from .dion3_oracle import (  # noqa: F401
    MUON_QUINTIC,
    num_selected,
    accumulate,
    row_l1,
    row_sumsq,
    select_rows,
    normalize,
    newton_schulz,
    round_to_bf16,
    round_to_fp32,
    decay_rows,
    update_rows,
    dion3_step,
    dion3_step_normuon,
    gram_newton_schulz,
    normuon_rows,
    normuon_update,
)
from .flops import (  # noqa: F401
    gram_ns_useful_flops,
    standard_ns_useful_flops,
    standard_ns_dense_flops,
)
