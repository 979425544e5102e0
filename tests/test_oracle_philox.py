"""Pins for the oracle's Philox-4x32-10 (oracle/philox.py).

Two independent references, neither of which is the oracle itself:
(a) the Random123 known-answer vectors (tests/golden/philox4x32_10_kat.txt);
(b) Triton's own ``tl.philox`` executed by its CPU interpreter (a third-party
    implementation run as a library, not copied).
"""

import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

from oracle.philox import philox4x32_10

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([int(t, 16) for t in line.split()])
    return rows


def test_known_answer_vectors():
    rows = _kat_rows()
    assert len(rows) == 3
    for r in rows:
        ctr, key, expect = r[0:4], r[4:6], r[6:10]
        out = philox4x32_10(*[np.array([c], dtype=np.uint32) for c in ctr], key[0], key[1])
        assert [int(o[0]) for o in out] == expect


def test_rounds_matter():
    # A plausible slip -- one round too few -- must change the output.
    import oracle.philox as ph
    saved = ph.PHILOX_ROUNDS
    try:
        ph.PHILOX_ROUNDS = 9
        out9 = [int(o[0]) for o in ph.philox4x32_10(*[np.zeros(1, np.uint32)] * 4, 0, 0)]
    finally:
        ph.PHILOX_ROUNDS = saved
    assert out9 != [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]


_TRITON_SCRIPT = textwrap.dedent(
    """
    import os, sys
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def kern(out_ptr, c0_ptr, c1_ptr, c2_ptr, c3_ptr, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        a, b, c, d = tl.philox(seed, tl.load(c0_ptr + i), tl.load(c1_ptr + i),
                               tl.load(c2_ptr + i), tl.load(c3_ptr + i))
        tl.store(out_ptr + 4 * i + 0, a)
        tl.store(out_ptr + 4 * i + 1, b)
        tl.store(out_ptr + 4 * i + 2, c)
        tl.store(out_ptr + 4 * i + 3, d)

    data = np.load(sys.argv[1])
    N = data["ctr"].shape[1]
    out = []
    for seed in data["seeds"]:
        o = torch.zeros(4 * N, dtype=torch.uint32)
        cs = [torch.from_numpy(data["ctr"][q].copy()) for q in range(4)]
        kern[(1,)](o, *cs, int(seed), N=N)
        out.append(o.numpy().reshape(N, 4).T.copy())
    np.save(sys.argv[2], np.stack(out))
    """
)


def test_matches_triton_interpreter(tmp_path):
    pytest.importorskip("triton")
    pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    N = 256
    ctr = rng.integers(0, 2**32, size=(4, N), dtype=np.uint64).astype(np.uint32)
    ctr[:, 0] = 0
    ctr[:, 1] = 0xFFFFFFFF
    seeds = np.array([0, 1234, 0xFFFFFFFFFFFFFFFF, 0x299F31D0A4093822,
                      int(rng.integers(0, 2**63))], dtype=np.uint64)
    src = tmp_path / "in.npz"
    dst = tmp_path / "out.npy"
    np.savez(src, ctr=ctr, seeds=seeds)
    script = tmp_path / "tri.py"
    script.write_text(_TRITON_SCRIPT)
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, str(script), str(src), str(dst)],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        pytest.skip("Triton interpreter unavailable: " + r.stderr.strip().splitlines()[-1])
    tri = np.load(dst)
    for s_i, seed in enumerate(seeds):
        seed = int(seed)
        ours = philox4x32_10(ctr[0], ctr[1], ctr[2], ctr[3], seed & 0xFFFFFFFF, seed >> 32)
        for q in range(4):
            np.testing.assert_array_equal(ours[q], tri[s_i, q])
