"""GB300-native (sm_103a) int4 routed-expert MoE layer: C-ABI library + thin Python binding.

    from int4_routed_expert_quantize_gb300 import coli
    layer = coli.MoeLayer(d=6144, f=2048, n_experts=256, top_k=8)
"""
