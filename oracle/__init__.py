"""CPU oracle for the DSA decode step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never calls
it, and it shares no code with the CUDA path: it imports nothing but numpy.

It is the plain definition of what the decode step computes, written out with
int64 integers and float64 reals, no blocking and no reordering:

* ``indexer_scores``  -- the lightning-indexer score of every visible cached
  position (the cost that grows with context on "ds4 glm53-m3ultra", page 1);
* ``topk_indices``    -- the k highest-scoring positions in a fixed order, by a
  full stable sort ("same positions selected, same order", page 1);
* ``sparse_attention`` -- softmax attention of every query head over the
  selected latent rows only (page 1: "roughly 2,048 selected positions");
* ``decode_step``     -- the three in sequence;
* ``indexer_front_end`` -- the indexer query and head weights of each row,
  projected from its hidden vector by 8-bit affine weights and quantised to the
  indexer's integer operands ("GLM-5.3-Flash-Alis-MLX-4bit", page 3: the
  indexer projections at 8 bits, groups of 64), with ``dequantize_affine``;
* ``e4m3_to_f64``     -- the FP8 E4M3 code of the FP8 latent cache
  ("glm53-tensorfold-spark", page 4: FP8 KV storage), decoded from the format's
  definition.

Readings where the pages are silent (each listed with its reason in the design
notes): the indexer applies a per-head ReLU before weighting by ``w`` and summing
over heads; indexer keys are one int8 vector per position shared by all heads;
ties are broken by the lower index; a row with at most k visible positions
selects all of them; the latent row is the key (all ``D_k`` columns) and its
first ``D_v`` columns are the value (absorbed MLA); indices are request-local.
"""
from .dsa import (  # noqa: F401
    indexer_scores,
    topk_indices,
    sparse_attention,
    attention_lse,
    decode_step,
    e4m3_to_f64,
    dequantize_affine,
    indexer_front_end,
    INT32_MIN,
    INT32_MAX,
)
