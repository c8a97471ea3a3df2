"""CPU oracle (test infrastructure only).

Only the tests, the package's smoke check and the bench's CPU-baseline leg may
import this package; the product path never does. See paged_kv.py.
"""
from .paged_kv import (copy_blocks, gather_request_kv, kv_range, paged_attention, resolve,
                       scatter_kv, softmax_attend, step)

__all__ = ["copy_blocks", "gather_request_kv", "kv_range", "paged_attention", "resolve",
           "scatter_kv", "softmax_attend", "step"]
