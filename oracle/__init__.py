"""CPU oracle for compressed-KV decode attention.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the decode path computes, written from the pages that
describe DeepSeek-V4's compressed attention.  Only the tests, the smoke check
in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.
The CUDA library never links, imports or calls anything here, and nothing here
imports the CUDA library or its Python binding.

Modules
-------
codecs     FP8 (e4m3 + e8m0 per 32), FP4 (e2m1 + e4m3 per 16) and bf16 row codecs; the
           index keys' page-split FP8 and Hadamard-rotated FP4 (e2m1 + e8m0 per 32)
expo       exp_own: the Cody-Waite exponential of the bit-exact compressor contract
rope       partial-RoPE tables (plain and YaRN) and rotations
compress   the gated per-channel pooling compressor (fp64 definition, fp32 contract)
indexer    lightning-indexer scores and top-k selection
attention  shared-KV sparse decode attention with window and sink
decode_state  the decode step's compressor state ring and window row

Precision: definitions run in fp64.  The one place that must be bit-exact
against the GPU - the bytes the compressor writes - is computed in the fp32
contract order spelled out in ``compress.py`` and ``expo.py``.

Every function is parity-pinned by the ``-m "not gpu"`` tests in ``tests/``
(worked examples the pages print, closed forms, library routines and brute
force); none of them is "parity unpinned".
"""
