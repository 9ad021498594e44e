"""Pins the oracle's parameter arithmetic against the counts the pages print."""
from oracle import moe_oracle as O


def _counts(golden):
    return {r[0]: float(r[1]) if "." in r[1] else int(r[1]) for r in golden("kimi_k2_param_counts.txt")}


def _cfg(golden):
    return {r[0]: r[1] for r in golden("kimi_k2_config.txt")}


def test_moe_block_count_from_model_totals(golden):
    n, c = _counts(golden), _cfg(golden)
    d, E, H = int(c["hidden_size"]), int(c["n_routed_experts"]), int(c["moe_intermediate_size"])
    S = int(c["n_shared_experts"])
    layers, dense = int(c["num_hidden_layers"]), int(c["first_k_dense_replace"])
    moe_layer = O.moe_layer_params(d, E, H, S)
    assert moe_layer == 16_958_226_816
    block = moe_layer + n["mla_attention"] + 2 * n["block_rmsnorm"]
    # the transformer blocks are one dense block and 60 MoE blocks
    assert (n["transformer_blocks"] - dense * n["dense_block"]) == (layers - dense) * block
    assert round(block / 1e9, 2) == n["largest_layer_billions"]
    assert (n["token_embedding"] + n["vocab_projection"] + n["transformer_blocks"]
            + n["final_rmsnorm"]) == n["model_total"]


def test_dense_swiglu_count(golden):
    n, c = _counts(golden), _cfg(golden)
    d, Hd = int(c["hidden_size"]), int(c["intermediate_size"])
    assert O.swiglu_params(d, Hd) == n["dense_swiglu_mlp"] == 396_361_728
    assert O.swiglu_params(d, Hd) / 2 ** 20 == n["dense_mlp_fp8_mib"]   # one byte per FP8 weight
    assert n["dense_block"] == n["mla_attention"] + 2 * n["block_rmsnorm"] + O.swiglu_params(d, Hd)


def test_active_parameter_count(golden):
    n, c = _counts(golden), _cfg(golden)
    d, E, H = int(c["hidden_size"]), int(c["n_routed_experts"]), int(c["moe_intermediate_size"])
    k, S = int(c["num_experts_per_tok"]), int(c["n_shared_experts"])
    layers, dense = int(c["num_hidden_layers"]), int(c["first_k_dense_replace"])
    active_moe = (k + S) * O.swiglu_params(d, H) + E * d + E
    active_block = active_moe + n["mla_attention"] + 2 * n["block_rmsnorm"]
    non_emb = (layers - dense) * active_block + dense * n["dense_block"] + n["final_rmsnorm"]
    assert round(non_emb / 1e9, 2) == n["active_non_embedding_billions"]
    with_emb = non_emb + n["token_embedding"] + n["vocab_projection"]
    assert round(with_emb / 1e9, 1) == n["active_with_embedding_billions"]
