"""Plain, slow, obviously-correct CPU oracle for the TurboQuant KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA library (``kv_cache_vector_head_gb300``) and
imports nothing from it.

Everything is computed in float64 (numpy / scipy); stored fields are rounded
to float32 exactly where the method stores them.  Each function cites the
passage of the source pages it follows.  Page titles are abbreviated:

* [Design study]   "TurboQuant Family Design Study for CPU and Browser WASM KV Caches"
* [Reconstruction] "Mathematical Reconstruction, Lineage, and Accuracy Limits of
                    TurboQuant and TurboVec"
* [README]         "TurboQuant: KV Cache Compression for LLM Inference" (README)

Where the pages are silent, garbled or lost (every formula of
[Reconstruction] is a lost image), the reading taken is stated at the
function; the list of readings lives in the repository design notes.

Modules
-------
codebook    Lloyd-Max codebook for the rotated-coordinate (sphere) marginal.
rng         SplitMix64 + Box-Muller: the oracle's own counter-based generator
            for the random draws of the method (rotation, signs, QJL matrix).
transforms  Dense Haar rotation (QR), Rademacher + FWHT rotation, QJL matrix.
codec       TurboQuant_prod (keys) and TurboQuant_mse (values) per vector,
            sign-magnitude bit-plane packing.
paging      Page sub-block layout, window policy, append state machine.
attention   Compressed-domain decode attention with an fp16 recent window.
"""

from . import codebook, rng, transforms, codec, paging, attention  # noqa: F401
