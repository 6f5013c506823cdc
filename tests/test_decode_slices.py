"""CPU-only checks of how the bf16 grouped decode kernel cuts its work list over its CTAs, through
the pa_debug_decode_slices hook (the same arithmetic the kernel runs): every unit belongs to
exactly one slice, the owner of a unit is the last slice that starts at or before it, the
slices are equal to within one unit except that the light ones are shorter by the deficit, and
with no light CTAs the cut is the plain equal one, slice c starting at floor(c U / C)."""
import os
import random
import shutil

import pytest

from paged_kv_cache_238_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists(
    os.path.join(ROOT, "paged_kv_cache_238_gb300", "libpa.so")), reason="needs nvcc to build libpa")


def _check(U, C, K, d):
    starts, owners = B.pa_debug_decode_slices(U, C, K, d)
    assert starts[0] == 0 and starts[C] == U
    assert all(a <= b for a, b in zip(starts, starts[1:]))
    # brute force: the owner of u is the last slice whose start is at or before u
    for u in range(U):
        c = owners[u]
        assert 0 <= c < C and starts[c] <= u and all(starts[x] > u for x in range(c + 1, C)), (U, C, K, d, u, c)
    sizes = [b - a for a, b in zip(starts, starts[1:])]
    active = 0 < K < C and d > 0 and U - (C - K) * d >= C
    if not active:
        assert starts == [c * U // C for c in range(C + 1)]
        return False
    full, light = sizes[:C - K], sizes[C - K:]
    assert min(sizes) >= 1                              # every slice keeps a unit
    assert max(full) - min(full) <= 1 and max(light) - min(light) <= 1
    # the light slices are shorter by the deficit (each slice rounds on its own)
    assert abs((sum(full) / len(full) - sum(light) / len(light)) - d) <= 1.0
    return True


@pytest.mark.parametrize("U,C,K,d", [
    (6122, 152, 15, 12),      # the GQA decode batch on a full GB300 grid
    (131072, 152, 15, 12),    # long split-KV
    (100, 152, 15, 12),       # fewer units than CTAs: equal slices, some empty
    (152, 152, 15, 12),       # one unit per CTA: the deficit does not fit
    (1, 1, 0, 0), (0, 7, 2, 3), (5000, 64, 6, 12), (5000, 120, 12, 12),
])
def test_slices_cases(U, C, K, d):
    _check(U, C, K, d)


def test_slices_random():
    rng = random.Random(20261203)
    n_active = 0
    for _ in range(400):
        C = rng.randint(1, 200)
        U = rng.randint(0, 4000)
        K = rng.randint(0, C)
        d = rng.randint(0, 40)
        n_active += _check(U, C, K, d)
    assert n_active > 100  # the light cut is exercised, not only the fallback


def test_slices_bad_arguments():
    with pytest.raises(B.PaError):
        B.pa_debug_decode_slices(-1, 8, 0, 0)
    with pytest.raises(B.PaError):
        B.pa_debug_decode_slices(10, 0, 0, 0)
