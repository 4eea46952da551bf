"""Seeded synthetic inputs (catalogues, model tensors, requests); no decoding arithmetic."""
from .generators import (CONFIGS, Config, DecoWeights, SynthModel, bf16_bits_to_f32, catalogue_dense_early,
                         catalogue_fixed_fanout, catalogue_uniform, catalogue_zipf_geometric,
                         catalogue_zipf_hier, distinct_per_group, f32_to_bf16_bits, make_catalogue,
                         make_concepts, make_deco, make_model, make_requests, product_catalogue, rng_for)

__all__ = [
    "CONFIGS", "Config", "DecoWeights", "SynthModel", "bf16_bits_to_f32", "catalogue_dense_early",
    "catalogue_fixed_fanout", "catalogue_uniform", "catalogue_zipf_geometric",
    "catalogue_zipf_hier", "distinct_per_group", "f32_to_bf16_bits", "make_catalogue",
    "make_concepts", "make_deco", "make_model", "make_requests", "product_catalogue", "rng_for",
]
