"""Oracle for the ReplaySSM decode path: a plain, slow, fp64 CPU restatement.

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The library
(``recurrent_state_decode_gb300``) never imports it, and it never imports the
library: the two share no code. Inputs arrive as numpy arrays (the exact bf16 /
fp32 values a GPU run sees, widened to fp64); every function returns fp64.

Sources, by page title and section:

* "ReplaySSM Caches Inputs Instead of State to Speed Up Hybrid-Model Decoding",
  section "How ReplaySSM works": the state is a checkpoint plus a buffer of the
  last L input records; non-flush steps compute the output from the checkpoint
  and the buffer without storing state; the L-th step folds the buffer into the
  checkpoint; outputs equal conventional decoding up to floating-point error.
* Same page, section "Why SSM layers slow down hybrid models": conventional
  decoding updates, reads and stores the full state every step; the SSM layers
  are Mamba-2 and Gated DeltaNet.
* "ReplaySSM" (the paper's code repository), introduction: cheap rollback by
  moving a buffer pointer; separate read and recurrence precisions.
* "ReplaySSM (a vLLM research fork)", section "Core implementation files":
  the kernel entry points (output-only AR step, state-and-output step,
  speculative decode on a circular buffer, cursor commit and reset).

The pages print no equations. The recurrences are the published Mamba-2
``selective_state_update`` decode step and the published gated delta rule;
the replay (unrolled) forms follow from them by algebra. Modules:

* ``mamba2``  -- conventional recurrence (the reference result) and the
  unrolled replay formula.
* ``gdn``     -- the same for Gated DeltaNet.
* ``kda``     -- the same for Kimi Delta Attention (the gated delta rule with
  a decay per key channel; the pages name the layer and give no equation).
* ``cursors`` -- integer model of the ring-buffer cursors.
* ``sessions`` -- runners of whole decode sessions (AR and speculative)
  with the conventional recurrence and the cursor model, producing every
  expected output, checkpoint and cursor.

Pins (in ``tests/test_oracle_*.py``): closed forms (A=0 cumulative sums,
pure-decay exponentials, skip path, delta-rule write/erase identities),
brute-force scalar unrolling of tiny states in extended precision, the replay
formula against the conventional recurrence, and hand-derived cursor traces.
"""
