"""Timed CPU baselines, reported beside the GPU figures by bench.py (never a
checker: parity is the oracle's job, in ``oracle/``).

  wsweep   Theorem 2.3's W-array grammar sweep and the direct CSR product, in
           C, sequential and OpenMP over the host cores.
"""
