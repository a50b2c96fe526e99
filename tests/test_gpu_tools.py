"""The measurement scripts run end to end on small cases: the multi-prefix sweep places what HOT
cannot hold in COLD (prefixes held by their requests are never evicted), and the prefill
benchmark reports a positive rate."""

import pytest

pytestmark = pytest.mark.gpu


def _flush():
    pass


def test_prefix_sweep_places_overflow_in_cold(cuda_ok):
    from shared_prefix_kv_decode_gb300 import prefix_sweep
    # HOT = 0.2 * 5120 = 1024 slots: two prefixes of 512 fit, the other two go to COLD
    out = prefix_sweep.measure(4, 512, 4, 2, _flush, 6800.0, n_slots=5120)
    assert out["hot_prefixes"] == 2 and out["cold_prefixes"] == 2
    assert out["cold_tokens_read"] == out["suffix_tokens"] + 2 * 512
    assert out["us_per_call"] > 0 and out["groups_dense"] == 2


def test_prefill_bench_runs(cuda_ok):
    from shared_prefix_kv_decode_gb300 import prefill_bench
    out = prefill_bench.measure(1024, 2, _flush, 1958.6)
    assert out["us_per_call"] > 0 and 0 < out["frac_of_measured_bf16"] < 1.5
