"""CPU oracle for the virtual-rank AllReduce -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow reference that the CUDA path is checked
against. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the library itself never does, and it
shares no code with the CUDA path (only the seeded input generator in
``ring_allreduce_reduction_gb300.workloads`` serves both).

Sources cited in this package:

* [Deep Dive] "NCCL Source Code Deep Dive: A GPU Journey of One AllReduce"
  (aireadcode.com, English edition; the Japanese edition carries the same
  chapters 1-4 and adds chapter 5, tuning, and chapter 6, enqueue).
* [Architecture] "NCCL architecture: topology, channels, algorithms and
  protocols" (arganzheng.life; part 4 of the series "Communication and
  interconnect: from NCCL to RDMA").

Modules:

* ``numerics``    element arithmetic: storage types, fp32-then-round ops,
                  the avg pre-scale and the integer avg post-op.
* ``schedule``    channel partition, loop/chunk addressing, ring
                  validation, binary and double binary trees.
* ``ring``        the ring AllReduce as a step machine with explicit FIFOs,
                  plus an independent association predictor.
* ``tree``        the double-binary-tree AllReduce (reduce up, broadcast
                  down).
* ``phases``      the reduce-scatter and all-gather phases of the ring run
                  alone (ReduceScatter, AllGather), with a predictor.
* ``closed_form`` the order-free definition (float64 / exact integers) and
                  the error bounds it is compared under.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force on tiny inputs, invariants and the
worked examples the pages print (``tests/golden/``).
"""
from . import numerics, schedule, ring, tree, phases, closed_form  # noqa: F401
from .ring import ring_allreduce, ring_predict  # noqa: F401
from .tree import tree_allreduce  # noqa: F401
