"""fp64 CPU oracle of the fused hidden-state KL loss: test infrastructure only (tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline legs). Never imported by the product."""
