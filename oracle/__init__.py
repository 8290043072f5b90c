"""Float64 CPU oracle for the DSA layer step (indexer -> exact top-k -> sparse MLA).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package: only
the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py`` may use it.  It shares no code with the CUDA
path; the two meet only at the byte layout of their inputs, which each side
implements on its own from the layout contract.

Source of the method: the vLLM blog post "vLLM delivers day-0 support for Kimi
K3.1 Pro", sections "Sparse Attention in K3.1 Pro" (indexer, top-2048, exact MLA
over the selected tokens), "KV cache footprint" (per-token byte table), "A KV
cache for three kinds of state" (packed per-block rows, page translation) and
"AMD / Quantization: Native MXFP4 indexer" (68-byte MXFP4 index keys).
"""
from .formats import (decode_e4m3, decode_e2m1, decode_e8m0, decode_bf16,
                      E4M3_TABLE, E2M1_TABLE)
from .dsa_oracle import (
    IDX_FP8, IDX_MXFP4, LAT_FP8, LAT_NVFP4, D_IDX, H_IDX, H_MLA, D_LAT, D_V,
    idx_bytes_per_token, lat_bytes_per_token, idx_page_bytes, lat_page_bytes,
    gather_index_keys, gather_latents, indexer_scores, indexer_scores_for_token,
    topk_select, sparse_mla, layer_step, decode_bytes_model, dense_mla_bytes,
    kv_bytes_per_token_all_layers,
)
