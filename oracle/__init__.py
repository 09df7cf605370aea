"""CPU fp64 oracle for Split-KV anchor attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
leg may import this package.  The product path (``lse_merge_gb300``) never
imports it, and it imports nothing from the product path: the two share only
the seeded input generators in ``workloads``.

Every function restates a definition from "Split-KV: Efficient Context
Parallelism for Training Diffusion Drafters" (Zhang, Zhang, Xie, Fan, You),
cited as [Split-KV §x, Eq. n / Fig. n].

Parity pins (see ``tests/test_oracle_pins.py``): every public function here is
pinned against something other than itself -- printed values of the worked
examples (Fig. 3, Fig. 5), closed forms, brute force, a library routine
(torch SDPA in fp64 with autograd) or finite differences.
"""
from .skv_oracle import *  # noqa: F401,F403
