"""Test infrastructure: the fp64 CPU oracle for LSH-sampled decode attention.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may import this
package. The product path (lsh_sampled_sparse_gb300) never imports it.
"""
from .magicpig_oracle import *  # noqa: F401,F403
