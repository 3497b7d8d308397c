"""Conservative DiT velocity-cache schedule: the oracle against the page's own
counts, and the library's host implementation against the oracle (no GPU)."""
import itertools
import os

import pytest

import rope_tfk_rmsnorm_gb300 as tfk
from oracle import velocity_cache
from rope_tfk_rmsnorm_gb300 import build as tfk_build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "velocity_cache_p1.txt")


def golden():
    kv = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=")
            kv[k] = float(v) if "." in v else int(v)
    return kv


@pytest.fixture(scope="module")
def lib():
    tfk_build.build()
    return tfk.load()


def test_oracle_reproduces_the_pages_counts():
    g = golden()
    s = velocity_cache.schedule(g["steps"], g["start_ratio"], g["end_ratio"], g["refresh_interval"],
                                g["max_consecutive_reuse"])
    assert sum(s) == g["cache_hits"]
    assert len(s) - sum(s) == g["cached_dit_calls"]
    # the cache off (an empty window) is the baseline: every step calls the DiT
    assert sum(velocity_cache.schedule(g["steps"], 0.0, 0.0)) == 0
    assert g["baseline_dit_calls"] == g["steps"]


def test_oracle_schedule_properties():
    s = velocity_cache.schedule(49)
    hits = [i for i, r in enumerate(s) if r]
    assert all(0.2 <= i / 49 < 0.8 for i in hits)               # only inside the window
    assert all(not (a and b) for a, b in zip(s, s[1:]))          # never two reuses in a row
    assert not s[0]                                              # nothing to reuse on step 0
    # a longer reuse budget is still capped by the refresh interval, and vice versa
    assert velocity_cache.schedule(49, refresh_interval=2, max_consecutive_reuse=3) == s
    assert velocity_cache.schedule(49, refresh_interval=5, max_consecutive_reuse=1) == s
    s3 = velocity_cache.schedule(49, refresh_interval=4, max_consecutive_reuse=3)
    assert sum(s3) > sum(s)


def _library_matches_oracle():
    g = golden()
    assert sum(tfk.tfk_velocity_cache_schedule(49)) == g["cache_hits"]
    for n, (a, b), ri, mr in itertools.product([0, 1, 2, 5, 10, 48, 49, 50, 100, 257],
                                               [(0.2, 0.8), (0.0, 1.0), (0.25, 0.75), (0.5, 0.5), (0.1, 0.3)],
                                               [1, 2, 3, 5], [0, 1, 2, 4]):
        assert tfk.tfk_velocity_cache_schedule(n, a, b, ri, mr) == velocity_cache.schedule(n, a, b, ri, mr), \
            (n, a, b, ri, mr)


def test_library_schedule_matches_the_oracle(lib):
    _library_matches_oracle()


@pytest.mark.gpu
def test_library_schedule_matches_the_oracle_on_the_gpu_host(lib):
    """The same check in the GPU run, where the library is built on the GPU host itself."""
    _library_matches_oracle()


def test_library_schedule_rejects_bad_arguments(lib):
    for args, words in [((-1, 0.2, 0.8, 2, 1), "num_steps = -1"), ((10, 0.8, 0.2, 2, 1), "<= end_ratio"),
                        ((10, -0.1, 0.8, 2, 1), "0 <= start_ratio"), ((10, 0.2, 1.5, 2, 1), "<= 1"),
                        ((10, 0.2, 0.8, 0, 1), "refresh_interval = 0"),
                        ((10, 0.2, 0.8, 2, -1), "max_consecutive_reuse = -1"),
                        ((10, float("nan"), 0.8, 2, 1), "finite")]:
        with pytest.raises(tfk.TfkError) as e:
            tfk.tfk_velocity_cache_schedule(*args)
        assert e.value.status == 1 and "tfk_velocity_cache_schedule" in str(e.value) and words in str(e.value), \
            (args, str(e.value))
