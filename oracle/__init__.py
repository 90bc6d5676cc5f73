"""CPU oracle for the compressed-KV decode-attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the ``libckv`` C ABI,
its kernels or the Python binding) may import, call, link or execute this
package.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.

The oracle is plain NumPy in float64.  Every function computes its result from
the definition the pages give (cited per function), with library primitives
(a matmul, a sort) as single steps and no blocking, fusion or reordering
beyond what the definition states.  It shares no code, table or constant
generator with the CUDA path.

Sources (titles of the pages, with the section each function follows):
  * "DeepSeek-V4 KV Cache 深度分析" -- appendix calculator, §二 (entry layout),
    §三 (CSA/HCA), §四 (indexer, its Hadamard rotation before FP4), §五
    (RoPE at the query and at the output, position -i), §六 (precision), §七
    (total formula), §十一 (forward flow chart).
  * "DeepSeek, KV 캐시를 토큰당 890바이트로 줄인 V4.1-Flash 공개" -- 핵심 내용
    (CSA2 modes, FP4 E2M1 + E4M3/16-channel main KV, the 2688 bound).
  * "KV cache 890 bajtów na token" -- "Trzy mechanizmy" (CSA2 Full / Reindex /
    Reuse, hierarchical indexer pool, FP4 main KV).
  * "DeepSeek V4 의 정확한 KV 캐시 사용량 분석" -- per-token byte arithmetic.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``.
The pages' 890 B/token figure for V4.1-Flash cannot be derived from what they
print, so no function computes it.
"""

from . import fp_formats, sizes, indexer, attention, csa2, rope, hadamard, paged  # noqa: F401
