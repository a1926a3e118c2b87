"""CPU oracle for the chunked KDA forward pass -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg use this
package.  The CUDA library never imports it.
"""
