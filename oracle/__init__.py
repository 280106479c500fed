"""CPU oracle for the paged GQA attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this package.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg
and its ``--impl reference`` arm) may import or run it.

It is plain, slow and deliberately direct: NumPy in float64, Python loops
where the method is a loop, every step written as the pages define it.  It
shares no code, table, constant or helper with the CUDA library; the two meet
only at the seeded inputs built by ``workloads``.

Modules
-------
paged_attention
    slot mapping, the KV scatter, varlen packing, gather-then-dense attention
    with the position-offset causal mask and GQA head sharing, decode.
sampler
    Philox4x32-10 (the counter-based generator both sides implement from its
    published definition), the exponential noise drawn from it, and the
    temperature sampler's exponential race.
rope
    rotary position embedding of Q and K before the KV write (V untouched).
"""
from . import paged_attention, rope, sampler  # noqa: F401
