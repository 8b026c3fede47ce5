"""fp64 CPU oracle of the KDA chunked forward.

TEST INFRASTRUCTURE ONLY. Only tests/, the smoke check in __graft_entry__.py and
the CPU-baseline leg of bench.py may import, call, link or run anything in this
package. The CUDA product path never does, and the two share no code: the only
thing both sides use is the seeded input generator module, which holds none of
the method's arithmetic.

Modules:
  kda_ref      plain fp64 token-by-token recurrence (numpy): the definition.
  kda_oracle.c the same definition in plain C, threaded over (sequence, head).
  c_oracle     ctypes front end of kda_oracle.c (builds it with gcc).
  chunked_ref  independent fp64 chunkwise (WY) form with exact pairwise decays;
               pins the token oracle and defines the per-chunk quantities.

Every function is pinned by tests under tests/ (test_oracle_pins.py) against
closed forms, invariants, special cases that reduce to library routines,
hand-derived golden values and brute force on tiny inputs.
"""
from .kda_ref import kda_fwd_ref, sigmoid, gate_log_decay, l2_normalize, to_f64  # noqa: F401
from .chunked_ref import kda_fwd_chunked, chunk_quantities, forward_substitution_inverse  # noqa: F401
