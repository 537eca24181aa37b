"""CPU oracle for one MoE layer's prefill -- TEST INFRASTRUCTURE.

Imported only by the tests, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline leg; the product library never touches it.
"""
from .oracle import (build, load, exp_f32, route_topk, route_csr,  # noqa: F401
                     grouped_placement, moe_layer_rows, num_threads, maxplus,
                     router_logits, down_scale_exp, q4_quantize, q4_dequantize)
