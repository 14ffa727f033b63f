"""The CPU oracle against what the Fathom page and the mathematics fix
(no GPU needed).  Each pin is described in ``tests/pins.py``."""
import pytest

from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(orc, pin):
    pin(orc)


def test_bytes_model_eq1():
    """Fathom page, section 1 and section 3.1 Eq. 1, for Qwen3-8B (36 layers,
    8 KV heads of 128 channels): dense bf16 KV 4.8 GB/step at 32k; a 136-bit scan
    reads 557 KB per (layer, head) pair at 32k, 160 MB/step at 32k and 5.1 GB at
    1M; winner rows are bounded by 2048 per KV head (k = 512, G = 4)."""
    from workload import bytes_model as bm
    L, H, D = 36, 8, 128
    assert round(bm.dense_kv_bytes(L, H, D, 32768) / 1e9, 1) == 4.8
    assert round(bm.scan_bytes(136, 32768) / 1e3) == 557
    assert round(bm.step_bytes(1, L, H, 136, 32768, 0) / 1e6) == 160
    assert round(bm.step_bytes(1, L, H, 136, 1 << 20, 0) / 1e9, 1) == 5.1
    assert bm.depth_bits([4] * 32 + [0] * 96) == 136
    assert bm.depth_bits([4] * 16 + [0] * 112) == 68
    assert bm.depth_bits([2] * 128) == 288
    assert bm.union_bound(4, 512) == 1940 <= 4 * 512
    # the row term does not grow with context, the scan term does
    a = bm.step_bytes(1, L, H, 136, 32768, 2048) - bm.step_bytes(1, L, H, 136, 32768, 0)
    b = bm.step_bytes(1, L, H, 136, 1 << 20, 2048) - bm.step_bytes(1, L, H, 136, 1 << 20, 0)
    assert a == b
