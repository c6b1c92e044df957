"""Batch-invariant paged-KV attention for one flat ragged step on GB300 (sm_103a).

The compute runs in the hand-written CUDA kernels of ``libpa.so``; this
package only marshals arguments (``invariant_paged_kv_gb300.pa``) and builds
seeded synthetic steps (``invariant_paged_kv_gb300.workload``).
"""
