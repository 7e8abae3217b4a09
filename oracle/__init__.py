"""CPU oracle of the int4 routed-expert MoE layer -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and the CPU-baseline leg of bench.py may import it."""
