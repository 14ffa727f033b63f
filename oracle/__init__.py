"""CPU oracle of the bit-plane KV scan path.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import it.  It shares no code
with the CUDA library in ``bit_plane_kv_encode_gb300``.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  or_fp16_bits / or_fp16_value : numpy float16 conversion (library routine).
  or_encode                    : exact rational floor of k/s per code; prefix of t
                                 planes = direct t-bit quantiser for t = 0..4;
                                 special values +a -> 15, -a -> 0, 0 -> 8; fixed
                                 bit-order fixture.
  or_dequant / or_scores       : full-depth scores = dot products with 4-bit
                                 dequantised keys built independently from k;
                                 depth-0 channels contribute exactly 0.
  or_alloc_depths              : brute-force enumeration of all 5^8 depth vectors
                                 at D = 8; uniform-g closed cases.
  or_fixed_depths              : brute-force ranking of summed |q|.
  or_topk                      : full Python sort on small n with ties.
  or_union                     : Python set union.
  or_attend / or_dense_attend  : textbook softmax attention in numpy; selection of
                                 all rows equals dense attention.
"""
from .oracle import Oracle, bf16_bits, build, load_variant  # noqa: F401
