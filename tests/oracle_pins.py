"""Checks that pin the oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:

* hand-derived golden vectors written out from the layout definition;
* an independent reading of the layout through numpy reshape/transpose;
* brute force over every range of tiny caches (with the round-trip and
  untouched-bytes invariants);
* the KV-cache capacity formula 2*B*S*H*D*P*N (capacity page);
* the worked transfer estimate of the disaggregation page (section 5.1).

They are plain functions so that ``test_oracle_pins.py`` can also run them
against deliberately broken copies of the oracle in a child process.
"""
from __future__ import annotations

import itertools
import sys
from dataclasses import replace
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

from synth.configs import Geometry, GEOMETRIES  # noqa: E402

GOLDEN = Path(__file__).resolve().parent / "golden"
_UINT = {1: np.uint8, 2: np.uint16, 4: np.uint32}


def read_golden(name):
    out = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        out[key.strip()] = val.strip()
    return out


def expand_runs(text):
    vals = []
    for tok in text.split():
        if ".." in tok:
            a, b = tok.split("..")
            vals.extend(range(int(a), int(b) + 1))
        else:
            vals.append(int(tok))
    return vals


def _geom_from(text, name="golden"):
    kv = dict(item.split("=") for item in text.split())
    return Geometry(name, int(kv["L"]), int(kv["B"]), int(kv["H"]), int(kv["D"]), int(kv["S"]),
                    int(kv["P"]), "raw")


def _fill(spec, n, dt):
    base = np.arange(n, dtype=np.int64)
    if spec == "iota":
        return base.astype(dt)
    if spec.startswith("iota+"):
        return (base + int(spec[5:])).astype(dt)
    raise ValueError(spec)


# ---- an independent reading of the layout ---------------------------------

def numpy_reading(g: Geometry, k: np.ndarray, v: np.ndarray, l0, l1, s, e) -> np.ndarray:
    """Pack through numpy views: K as [L,B,H,D/x,S,x] -> [L,B,H,S,D] by a
    transpose, V as [L,B,H,S,D]; slices laid end to end in the order
    layer, K/V, sequence, head, token, d."""
    dt = _UINT[g.elem_bytes]
    L, B, H, D, S = g.num_layers, g.batch, g.num_heads, g.head_dim, g.max_seq
    x = 16 // g.elem_bytes
    dense = B * H * D * S
    kk = (k.view(dt).reshape(L, g.layer_elems)[:, :dense]
          .reshape(L, B, H, D // x, S, x).transpose(0, 1, 2, 4, 3, 5).reshape(L, B, H, S, D))
    vv = v.view(dt).reshape(L, g.layer_elems)[:, :dense].reshape(L, B, H, S, D)
    parts = [np.zeros(0, dt)]
    for l in range(l0, l1):
        for X in (kk, vv):
            for b in range(B):
                parts.append(X[l, b, :, s[b]:e[b], :].reshape(-1))
    return np.concatenate(parts).view(np.uint8)


def selected_mask(g: Geometry, l0, l1, s, e):
    """Boolean element masks of K and V marking the selected slices."""
    L, B, H, D, S = g.num_layers, g.batch, g.num_heads, g.head_dim, g.max_seq
    x = 16 // g.elem_bytes
    dense = B * H * D * S
    mk = np.zeros((L, g.layer_elems), bool)
    mv = np.zeros((L, g.layer_elems), bool)
    mk5 = mk[:, :dense].reshape(L, B, H, D // x, S, x)
    mv5 = mv[:, :dense].reshape(L, B, H, S, D)
    for b in range(B):
        mk5[l0:l1, b, :, :, s[b]:e[b], :] = True
        mv5[l0:l1, b, :, s[b]:e[b], :] = True
    return mk.reshape(-1), mv.reshape(-1)


def random_cache(g: Geometry, rng):
    k = rng.integers(0, 256, size=g.tensor_bytes, dtype=np.uint8)
    v = rng.integers(0, 256, size=g.tensor_bytes, dtype=np.uint8)
    return k, v


def random_ranges(g: Geometry, rng, allow_empty=True):
    s = np.zeros(g.batch, np.int32)
    e = np.zeros(g.batch, np.int32)
    for b in range(g.batch):
        a, c = sorted(rng.integers(0, g.max_seq + 1, size=2))
        if not allow_empty and a == c:
            c = min(g.max_seq, a + 1)
            a = c - 1
        s[b], e[b] = a, c
    return s, e


# ---- pins -------------------------------------------------------------------

def pin_golden(orc, name):
    gd = read_golden(name)
    g = _geom_from(gd["geometry"])
    dt = _UINT[g.elem_bytes]
    k = _fill(gd["k_fill"], g.tensor_elems, dt).view(np.uint8)
    v = _fill(gd["v_fill"], g.tensor_elems, dt).view(np.uint8)
    l0, l1 = (int(t) for t in gd["layers"].split())
    s = np.array(gd["seq_start"].split(), np.int32)
    e = np.array(gd["seq_end"].split(), np.int32)
    want = np.array(expand_runs(gd["staging"]), dt)
    got = orc.pack(g, k, v, l0, l1, s, e).view(dt)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.array_equal(got, want), (name, got, want)
    # the unpack of the golden staging into a zeroed cache puts every value back
    k2 = np.zeros_like(k)
    v2 = np.zeros_like(v)
    orc.unpack(g, k2, v2, l0, l1, s, e, want.view(np.uint8))
    mk, mv = selected_mask(g, l0, l1, s, e)
    assert np.array_equal(k2.view(dt)[mk], k.view(dt)[mk])
    assert np.array_equal(v2.view(dt)[mv], v.view(dt)[mv])
    assert not k2.view(dt)[~mk].any() and not v2.view(dt)[~mv].any()


READING_GEOMS = [
    Geometry("r1", 2, 3, 2, 16, 9, 2, "raw"),
    Geometry("r2", 3, 2, 3, 32, 7, 2, "raw"),
    Geometry("r3", 1, 2, 2, 48, 5, 2, "raw"),           # D/x = 6, not a power of two
    Geometry("r4", 2, 2, 1, 32, 6, 1, "raw"),           # 1-byte elements, x = 16
    Geometry("r5", 2, 1, 2, 8, 5, 4, "raw"),            # 4-byte elements, x = 4
    Geometry("r6", 2, 2, 2, 16, 4, 2, "raw", layer_stride_elems=2 * 2 * 16 * 4 + 24),
]


def pin_numpy_reading(orc, trials=6, seed=7):
    rng = np.random.default_rng(seed)
    for g in READING_GEOMS:
        k, v = random_cache(g, rng)
        for _ in range(trials):
            s, e = random_ranges(g, rng)
            l0 = int(rng.integers(0, g.num_layers + 1))
            l1 = int(rng.integers(l0, g.num_layers + 1))
            want = numpy_reading(g, k, v, l0, l1, s, e)
            got = orc.pack(g, k, v, l0, l1, s, e)
            assert np.array_equal(got, want), (g.name, l0, l1, s, e)


def pin_brute_force(orc):
    """Every range pair of a 2-sequence cache with S = 4, every layer range."""
    g = Geometry("bf", 2, 2, 2, 16, 4, 2, "raw")
    rng = np.random.default_rng(11)
    k, v = random_cache(g, rng)
    pairs = [(a, c) for a in range(g.max_seq + 1) for c in range(a, g.max_seq + 1)]
    sentinel = np.uint8(0xA5)
    for (l0, l1) in [(0, 2), (1, 2), (0, 1), (1, 1)]:
        for (r0, r1) in itertools.product(pairs, pairs):
            s = np.array([r0[0], r1[0]], np.int32)
            e = np.array([r0[1], r1[1]], np.int32)
            want = numpy_reading(g, k, v, l0, l1, s, e)
            got = orc.pack(g, k, v, l0, l1, s, e)
            assert np.array_equal(got, want), (l0, l1, s, e)
            k2 = np.full_like(k, sentinel)
            v2 = np.full_like(v, sentinel)
            orc.unpack(g, k2, v2, l0, l1, s, e, got)
            mk, mv = selected_mask(g, l0, l1, s, e)
            mkb = np.repeat(mk, g.elem_bytes)
            mvb = np.repeat(mv, g.elem_bytes)
            assert np.array_equal(k2[mkb], k[mkb]) and np.array_equal(v2[mvb], v[mvb])
            assert (k2[~mkb] == sentinel).all() and (v2[~mvb] == sentinel).all()


def pin_capacity_formula(orc):
    """Full-prompt staging size equals 2*B*S*H*D*P*N (capacity page)."""
    for g in GEOMETRIES + READING_GEOMS:
        s = np.zeros(g.batch, np.int32)
        e = np.full(g.batch, g.max_seq, np.int32)
        n = g.num_layers
        formula = 2 * g.batch * g.max_seq * g.num_heads * g.head_dim * g.elem_bytes * n
        assert orc.staging_bytes(g, 0, n, s, e) == formula, g.name
    gd = read_golden("kv_capacity_page_example.txt")
    for key, ctx in (("context_100000", 100000), ("context_102400", 102400)):
        g = Geometry("cap", int(gd["layers"]), int(gd["batch"]), int(gd["heads"]),
                     int(gd["head_dim"]), ctx, int(gd["elem_bytes"]), "bf16")
        s = np.zeros(g.batch, np.int32)
        e = np.full(g.batch, ctx, np.int32)
        assert orc.staging_bytes(g, 0, g.num_layers, s, e) == int(gd[key])
    # the bytes actually written by a full pack of a small cache
    g = READING_GEOMS[0]
    rng = np.random.default_rng(3)
    k, v = random_cache(g, rng)
    s = np.zeros(g.batch, np.int32)
    e = np.full(g.batch, g.max_seq, np.int32)
    out = orc.pack(g, k, v, 0, g.num_layers, s, e)
    assert out.size == 2 * g.batch * g.max_seq * g.num_heads * g.head_dim * g.elem_bytes * \
        g.num_layers


def pin_distserve_example(orc):
    """4.5 MB per token of OPT-175B and 17.6 ms for 2048 tokens over 8x64 GB/s
    (disaggregation page, section 5.1)."""
    gd = read_golden("distserve_opt175b.txt")
    tokens = int(gd["tokens"])
    g = Geometry("opt175b", int(gd["model_layers"]), 1, int(gd["model_heads"]),
                 int(gd["model_head_dim"]), tokens, int(gd["elem_bytes"]), "fp16")
    one = orc.staging_bytes(g, 0, g.num_layers, np.array([0], np.int32), np.array([1], np.int32))
    assert one == float(gd["mb_per_token"]) * 2 ** 20, one
    total = orc.staging_bytes(g, 0, g.num_layers, np.array([0], np.int32),
                              np.array([tokens], np.int32))
    ms = total / (int(gd["links"]) * int(gd["link_gbs"]) * 2 ** 30) * 1e3
    assert abs(ms - float(gd["latency_ms"])) < 0.05, ms


def pin_source_of(orc):
    """The sampled-lookup walk agrees with the full pack at every offset."""
    rng = np.random.default_rng(5)
    for g in READING_GEOMS[:4]:
        k, v = random_cache(g, rng)
        s, e = random_ranges(g, rng)
        want = numpy_reading(g, k, v, 0, g.num_layers, s, e)
        dt = _UINT[g.elem_bytes]
        n = want.size // g.elem_bytes
        kv, idx = orc.source_of(g, 0, g.num_layers, s, e, np.arange(n))
        vals = np.where(kv == 0, k.view(dt)[idx], v.view(dt)[idx])
        assert np.array_equal(vals.astype(dt), want.view(dt)), g.name


ALL_PINS = [
    lambda o: pin_golden(o, "pack_single_head_iota.txt"),
    lambda o: pin_golden(o, "pack_multi_iota.txt"),
    pin_numpy_reading,
    pin_brute_force,
    pin_capacity_formula,
    pin_distserve_example,
    pin_source_of,
]


def run_all_pins(lib_path: str) -> int:
    """Run every pin against the oracle compiled at ``lib_path``; return the
    number of pins that failed."""
    import oracle
    orc = oracle.Oracle(oracle.load(Path(lib_path)))
    failed = 0
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failed += 1
    return failed


if __name__ == "__main__":
    sys.exit(min(run_all_pins(sys.argv[1]), 100))
