"""CPU oracle of the chunk-bounded top-k softmax MoE block.

TEST INFRASTRUCTURE ONLY: only tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py may import it.  The product path never does.
"""
