"""CPU oracle for PaTH causal attention — test infrastructure only.

Importable by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg;
the CUDA package never imports it.
"""
