"""Plain fp64 CPU oracle for absorbed-MLA decode attention (over a bf16 or an
FP8 latent cache), the weight-absorption BMMs on either side of it, and the
sparse-attention indexer (token scores, top-k lists).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library, its
Python binding, the timed legs of the benchmark) may import or call this
package; only the test-suite, the smoke check and the benchmark's CPU-baseline
and reference legs do.  It shares no code with the GPU implementation.
"""

from .mla_oracle import (  # noqa: F401
    D_QK,
    D_V,
    PAGE,
    attend,
    bf16_bits_to_f64,
    combine,
    f64_to_bf16_bits,
    mla_decode,
    physical_rows,
    softmax_weights,
    visible_positions,
)
from .absorb_oracle import absorb_o, absorb_q  # noqa: F401,E402
from .indexer_oracle import indexer_scores, indexer_topk, topk_select, topk_select_fast  # noqa: F401,E402
from .fp8_oracle import e4m3_to_f64, fp8_rows_to_f64, mla_decode_fp8, ue8m0_to_f64  # noqa: F401,E402
