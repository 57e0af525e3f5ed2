"""CPU oracle for speculative-decoding verification and D-cut depth scheduling.

TEST INFRASTRUCTURE ONLY.  Plain, slow, fp64 numpy restatement of what the
method computes, written from the pages' description of the method:

  * "AngelSpec explainer" = the article "AngelSpec: specialize the drafter,
    share the verification budget" (ai.thesatyajit.com/articles/angelspec).
  * "AngelSpec release article" = the tradepoint.io news article on the
    open-source release of AngelSpec.
  * "AngelSpec abstract" = the abstract of "AngelSpec: Towards Real-World High
    Performance Inference with Speculative Decoding" (Liu et al., Tencent).

Only tests/, the package's smoke() entry point and bench.py's CPU-baseline leg
may import this package.  It shares no code with the CUDA library and imports
nothing from it.  Every function here is pinned by a `-m "not gpu"` test
against something other than itself (library routines, closed forms, exact
enumeration, printed values), except where its docstring says
"parity unpinned".
"""
from .philox import philox4x32_10, uniform, PURPOSE_ACCEPT, PURPOSE_RESAMPLE, PURPOSE_DRAFT
from .verify import (softmax_T, verify_request, verify_batch, request_uniforms, decode_rows,
                     NEAR_ACCEPT, NEAR_PICK)
from .schedule import (prefix_confidences, k_rho, candidate_budgets, dcut_schedule, table_cost,
                       check_cost_table)
from .metrics import mean_accepted_length, mean_acceptance, expected_accept_len
from .tree import verify_tree, verify_tree_batch, children_of
