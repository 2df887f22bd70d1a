"""CPU oracle for absorbed MLA decode over a paged latent cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it. The
CUDA library never calls into it and shares no code with it.
"""

from .mla_oracle import (  # noqa: F401
    absorb_query,
    dcp_combine,
    dcp_decode_partials,
    dcp_local_seq_lens,
    dcp_owner,
    dequantize_e4m3_cache,
    e4m3_to_float,
    gather_request_latent,
    merge_partials,
    mha_compute_friendly,
    mla_decode_multi_token_reference,
    mla_decode_reference,
    mla_decode_reference_fp8,
    mla_decode_split_partials,
    q_absorb_concat_cache,
    split_token_ranges,
    up_project,
    v_up_proj,
)
