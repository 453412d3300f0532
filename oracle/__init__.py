"""Float64 CPU oracle for the adapted linear layer in normal form.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA path (kernels, headers, helpers, tables) and never
reads a value produced by it; the only module both sides import is the seeded
input generator ``workloads``, which holds none of the method's arithmetic.

It is a plain, slow, obviously-correct restatement of what the article
"Scute: Exact Batched Serving for PEFT Adapters Beyond LoRA" (paper-daily.com;
cited below as *the article*) says the layer computes, in float64 with NumPy:

* ``methods``      each PEFT method from its own definition;
* ``normal_form``  the six-slot normal form, the method -> slot mapping, the
                   fold rule applied at load, and the merged per-adapter weight;
* ``indexing``     the token -> segment indexing (stable sort by method, id);
* ``batch``        a heterogeneous batch evaluated row by row group;
* ``byte_model``   the byte count of one call, from its definition.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against hand-derived worked examples (``tests/golden/``), closed forms,
invariants, library special cases and brute force.  The end-to-end numbers are
not pinned by any value the article prints (it prints no worked example).
"""
from . import methods, normal_form, indexing, batch, byte_model  # noqa: F401
