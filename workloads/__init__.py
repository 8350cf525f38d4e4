"""Seeded synthetic inputs for the paged-KV hot path.

This module builds INPUTS only (queries, new and cached K/V values, slots,
block tables, staged table diffs); it holds none of the arithmetic of the
method, and is the one module that both the CUDA path's tests/benchmark and
the CPU oracle draw their inputs from.

Shapes follow the workloads of the pages, at one attention layer:
  1 "tiny decode"        4 requests, contexts {17,33,64,100}, 4/4 heads, D 64, B 16,
                         64-block pool with random placement, scale 1/8.
  2 "decode 7B-like"     256 requests, 32/32 heads, D 128, B 16, context U[128,2048],
                         pool = exactly the blocks needed, tables a random permutation.
  3 "mixed chunked"      64 decodes (context U[1024,4096]) + prefill chunks of
                         1024/1024/1920 tokens after cached prefixes of 0/2048/8192,
                         causal, 32/8 heads (GQA), D 128, B 16 (4032 tokens <= 4096).
  4 "prefix-shared"      8 groups x 16 samples sharing one 2048-token prompt, private
                         tails U[0,512], 1-token decode, 32/8 heads, D 128, B 16, FP8 KV.
  5 "long context"       32 requests of 32768 tokens, 64/8 heads, D 128, B 64; every
                         4th request runs a 2048-token chunk at the end of its
                         context, the others decode one token; bf16 or FP8 KV.
Values are N(0,1) rounded to bf16. Structure (lengths, placements, slots) comes
from numpy's PCG64 with the given seed; bulk values come from a torch generator
on the requested device with the same seed, so large workloads are generated
where they will be used.

Cache state before the step: every token before the step's query tokens is
already stored (``ctx_*``); the step's own tokens (``new_*``) are written by the
step. Unused pool cells hold NaN (bf16 0x7FC0 / E4M3 0x7F) so that a read of a
cell that the method must not see shows up as NaN.
"""
from .generate import (CONFIG_NAMES, Workload, build, make, staged_diffs_from_tables,
                       config_seed)

__all__ = ["CONFIG_NAMES", "Workload", "build", "make", "staged_diffs_from_tables",
           "config_seed"]
