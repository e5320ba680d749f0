"""CPU oracle for selective KV-cache refresh.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
baseline / reference legs of bench.py may import anything from this package.
The product path (libkvr and its Python binding) never imports it, and it
imports nothing from the product path: the two share no code.  The only
module both sides consume is selective_kv_cache_gb300.workloads, which draws
seeded random inputs and holds none of the method's arithmetic.

Everything is plain numpy in float64, one step per definition on the pages,
with rounding to the model's storage dtype only where a tensor is stored
(see refresh.round_store).
"""
from .refresh import *  # noqa: F401,F403
from .select import *   # noqa: F401,F403
from . import policy  # noqa: F401  (CacheReforge layer-range policy: oracle.policy.*)
from . import sur  # noqa: F401  (Semantic-Unit Refresh selection: oracle.sur.*)
