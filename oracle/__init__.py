"""fp64 CPU oracle for split-KV paged decode attention (test infrastructure only)."""
from .splitkv_oracle import *  # noqa: F401,F403
from .splitkv_oracle import (MAX_SPLITS, ITEM_OVERHEAD, COMBINE_COST, MAX_WAVES,  # noqa: F401
                             _makespan)
