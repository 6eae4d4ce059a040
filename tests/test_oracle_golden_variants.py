"""The oracle's sinks, sliding window, ALiBi and sqrt ALiBi against the
hand-worked three-key decode in tests/golden/variants_decode.txt (CPU only)."""
import math
import os

import numpy as np
import pytest

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "variants_decode.txt")


def _load():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


V = _load()


def _run(**kw):
    q = np.array([[V["q"]]], np.float32)                                   # [T=1, H=1, D=2]
    kc = np.zeros((1, 4, 1, 2), np.float32)
    vc = np.zeros((1, 4, 1, 2), np.float32)
    for j in range(3):
        kc[0, j, 0], vc[0, j, 0] = V[f"k{j}"], V[f"v{j}"]
    kc[0, 3], vc[0, 3] = np.nan, np.nan                                    # never read
    return orc.paged_attention(q, kc, vc, np.array([[0]], np.int32), np.array([3], np.int32),
                               np.array([0, 1], np.int32), 1, 1, 2, 4, 1.0, **kw)[0, 0]


@pytest.mark.parametrize("name,kw", [
    ("plain", {}),
    ("sink0", dict(sinks=np.array([0.0]))),
    ("window2", dict(sliding_window=2)),
    ("alibi_ln2", dict(alibi_slopes=np.array([math.log(2.0)]))),
    ("alibi_sqrt_ln2", dict(alibi_slopes=np.array([math.log(2.0)]), alibi_sqrt=True)),
])
def test_hand_worked_variant(name, kw):
    np.testing.assert_allclose(_run(**kw), V[name], rtol=0, atol=1e-14)
