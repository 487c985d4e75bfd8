"""Pins for the oracle's Philox4x32-10 and its uniform.

The oracle's generator is checked against an independent library
implementation of the same published generator (Salmon et al., SC'11): the
``tl.philox`` routine of Triton, run by Triton's CPU interpreter in a child
process.  Not a GPU test: the interpreter executes on the host.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle

CASES = [
    ((0, 0, 0, 0), (0, 0)),
    ((1, 0, 0, 0), (0, 0)),
    ((0, 1, 2, 3), (7, 0)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0)),
    ((5, 1, 63, 12345), (0xDEADBEEF, 0x12345678)),
]

_CHILD = r"""
import json, os, sys
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl
@triton.jit
def k(out_ptr, seed, c0, c1, c2, c3):
    a, b, c, d = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + 0, a); tl.store(out_ptr + 1, b)
    tl.store(out_ptr + 2, c); tl.store(out_ptr + 3, d)
res = []
for ctr, key in json.loads(sys.argv[1]):
    o = torch.zeros(4, dtype=torch.int32)
    seed = key[0] | (key[1] << 32)
    if seed >= 2**63:
        seed -= 2**64
    k[(1,)](o, seed, *[c - 2**32 if c >= 2**31 else c for c in ctr])
    res.append([x & 0xFFFFFFFF for x in o.tolist()])
print(json.dumps(res))
"""


def _triton_philox(cases):
    pytest.importorskip("triton")
    env = dict(os.environ, TRITON_INTERPRET="1")
    out = subprocess.run([sys.executable, "-c", _CHILD, json.dumps(cases)],
                         env=env, capture_output=True, text=True, timeout=300)
    if out.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + out.stderr[-300:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_philox_matches_library_generator():
    ref = _triton_philox([[list(c), list(k)] for c, k in CASES])
    for (ctr, key), want in zip(CASES, ref):
        got = oracle.philox4x32_10(ctr, key).tolist()
        assert got == want, (ctr, key, [hex(x) for x in got], [hex(x) for x in want])


def test_u24_is_top_bits_of_first_word():
    for seed, step, seq, pos, draw in [(0, 0, 0, 0, 0), (3, 7, 11, 2, 1), (2**40 + 5, 2**33 + 9, 255, 6, 1)]:
        ctr = [pos, draw, seq, step & 0xFFFFFFFF]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        assert oracle.u24(seed, step, seq, pos, draw) == int(oracle.philox4x32_10(ctr, key)[0]) >> 8


def test_u24_uniformity():
    # 2^16 draws over (seq, pos): 64-bin chi-square well inside its 99.9% bound
    from scipy.stats import chi2
    u = np.array([oracle.u24(11, 3, s, p, 0) for s in range(4096) for p in range(16)], np.float64)
    u = u / 2**24
    assert u.min() >= 0 and u.max() <= 1 - 2**-24
    h, _ = np.histogram(u, bins=64, range=(0, 1))
    e = u.size / 64
    assert ((h - e) ** 2 / e).sum() < chi2.ppf(0.999, 63)
    # distinct draws differ (counter words are all used)
    a = {oracle.u24(1, 0, 0, 0, d) for d in range(4)}
    b = {oracle.u24(1, s, 0, 0, 0) for s in range(4)}
    assert len(a) == 4 and len(b) == 4
