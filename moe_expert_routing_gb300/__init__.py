"""GB300-native per-layer MoE block: exact routing, expert union, 4-bit SwiGLU experts, combine.

The compute path is the CUDA library ``libsmoe.so`` (C ABI declared in ``include/smoe.h``);
``moe_expert_routing_gb300.smoe`` is its thin Python binding and
``moe_expert_routing_gb300.workload`` the seeded synthetic input generator.  Importing the
package loads neither the library nor torch's CUDA context.
"""
