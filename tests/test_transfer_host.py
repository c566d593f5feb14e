"""Host-side logic of the transfer staging (no GPU)."""
from paged_decode_attention_02_gb300 import transfer as tr


def test_choose_granularity_threshold():
    assert tr.choose_granularity(100, 2048) == "request"
    assert tr.choose_granularity(2047, 2048) == "request"
    assert tr.choose_granularity(2048, 2048) == "layer"
    assert tr.choose_granularity(10 ** 6, 2048) == "layer"
