"""The oracle against what the pages and the layout definition fix (CPU)."""
import os
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest

import oracle
from synth.configs import Geometry
from tests import oracle_pins as P

ORC = oracle.default()


def test_golden_single_head():
    P.pin_golden(ORC, "pack_single_head_iota.txt")


def test_golden_multi_layer_sequence_head():
    P.pin_golden(ORC, "pack_multi_iota.txt")


def test_numpy_layout_reading():
    P.pin_numpy_reading(ORC)


def test_brute_force_every_range():
    P.pin_brute_force(ORC)


def test_capacity_formula():
    P.pin_capacity_formula(ORC)


def test_distserve_worked_example():
    P.pin_distserve_example(ORC)


def test_sampled_lookup_matches_pack():
    P.pin_source_of(ORC)


def test_roundtrip_and_untouched_medium():
    g = Geometry("m", 3, 4, 3, 64, 40, 2, "raw")
    rng = np.random.default_rng(21)
    k, v = P.random_cache(g, rng)
    for _ in range(4):
        s, e = P.random_ranges(g, rng)
        st = ORC.pack(g, k, v, 1, 3, s, e)
        k2 = np.full_like(k, 0x5A)
        v2 = np.full_like(v, 0x5A)
        ORC.unpack(g, k2, v2, 1, 3, s, e, st)
        mk, mv = P.selected_mask(g, 1, 3, s, e)
        mk = np.repeat(mk, 2)
        mv = np.repeat(mv, 2)
        assert np.array_equal(k2[mk], k[mk]) and np.array_equal(v2[mv], v[mv])
        assert (k2[~mk] == 0x5A).all() and (v2[~mv] == 0x5A).all()


def test_stream_layers_equals_swap_out():
    """Layer-by-layer streaming (Fig 7b) leaves the same host bytes as one
    swap-out of the same layers."""
    g = Geometry("m", 4, 3, 2, 32, 20, 2, "raw")
    rng = np.random.default_rng(22)
    k, v = P.random_cache(g, rng)
    s, e = P.random_ranges(g, rng)
    assert np.array_equal(ORC.stream_layers(g, k, v, 0, 4, s, e),
                          ORC.swap_out(g, k, v, 0, 4, s, e))


def test_snapshot_plus_deltas_restore():
    """Replica = snapshot of [0,len0) + one-token deltas; restoring them in
    order into a zeroed cache gives the live cache on the covered tokens
    (state replication and recovery, Fig 10)."""
    g = Geometry("m", 2, 3, 2, 16, 12, 2, "raw")
    rng = np.random.default_rng(23)
    k, v = P.random_cache(g, rng)
    len0 = np.array([3, 5, 1], np.int32)
    recs = [(0, 2, np.zeros(3, np.int32), len0,
             ORC.pack(g, k, v, 0, 2, np.zeros(3, np.int32), len0))]
    pos = len0.copy()
    for step in range(4):
        s = pos.copy()
        e = pos + np.array([1, 1, 1 if step < 2 else 0], np.int32)  # seq 2 finishes
        recs.append((0, 2, s, e, ORC.pack(g, k, v, 0, 2, s, e)))
        pos = e
    k2, v2 = ORC.restore(g, recs)
    mk, mv = P.selected_mask(g, 0, 2, np.zeros(3, np.int32), pos)
    mk = np.repeat(mk, 2)
    mv = np.repeat(mv, 2)
    assert np.array_equal(k2[mk], k[mk]) and np.array_equal(v2[mv], v[mv])
    assert not k2[~mk].any() and not v2[~mv].any()


def test_rejects_bad_arguments():
    g = Geometry("m", 2, 2, 2, 16, 8, 2, "raw")
    ok = (np.zeros(2, np.int32), np.full(2, 8, np.int32))
    assert ORC.check(g, 0, 2, *ok) == 0
    assert ORC.check(g, 0, 3, *ok) != 0
    assert ORC.check(g, 1, 0, *ok) != 0
    assert ORC.check(g, 0, 2, np.array([3, 0], np.int32), np.array([2, 8], np.int32)) != 0
    assert ORC.check(g, 0, 2, np.array([0, 0], np.int32), np.array([9, 8], np.int32)) != 0
    bad_d = Geometry("m", 2, 2, 2, 12, 8, 2, "raw")  # D not a multiple of x = 8
    assert ORC.check(bad_d, 0, 2, *ok) != 0


# ---- the pins have teeth: each planted mistake fails at least one pin -------
MUTANTS = {
    "chunk_lane_split": ("* (D / x) + d / x) * S + t) * x + d % x",
                         "* (D / x) + d % (D / x)) * S + t) * x + d / (D / x)"),
    "v_read_as_k": ("return l * layer_stride + ((b * H + h) * S + t) * D + d;",
                    "return l * layer_stride + (((b * H + h) * (D / 8) + d / 8) * S + t) * 8 + d % 8;"),
    "k_then_v_swapped": ("kv == 0 ?", "kv == 1 ?"),
    "sequence_head_transposed": ("(b * H + h)", "(h * B + b)"),
    "layer_stride_dropped": ("return l * layer_stride +", "return 0 * l * layer_stride +"),
    "token_off_by_one": ("for (int64_t t = seq_start[b]; t < seq_end[b]; ++t)",
                         "for (int64_t t = seq_start[b] + (seq_start[b] < seq_end[b] && seq_end[b] < S); t < seq_end[b] + (seq_start[b] < seq_end[b] && seq_end[b] < S); ++t)"),
    "d_reversed": ("const int64_t x = 16 / P;\n  int64_t off = 0;",
                   "const int64_t x = 16 / P;\n  int64_t off = 0;\n  const int64_t dflip = D - 1;"),
    # unpack alone writes V slices into K (pack untouched)
    "unpack_v_into_k": ("uint8_t* dst =\n                  kv == 0 ?",
                        "uint8_t* dst =\n                  kv >= 0 ?"),
    # layer and K/V loops exchanged in pack and unpack alike (round trips still hold)
    "layer_inside_kv": ("for (int64_t l = l0; l < l1; ++l)\n    for (int kv = 0; kv < 2; ++kv)",
                        "for (int kv = 0; kv < 2; ++kv)\n    for (int64_t l = l0; l < l1; ++l)"),
    # sequence and head loops exchanged in pack and unpack alike
    "head_outside_sequence": ("      for (int64_t b = 0; b < B; ++b)\n        for (int64_t h = 0; h < H; ++h)\n          for (int64_t t",
                              "      for (int64_t h = 0; h < H; ++h)\n        for (int64_t b = 0; b < B; ++b)\n          for (int64_t t"),
    # the size formula without its factor 2 (K and V)
    "size_without_kv": ("return 2 * (int64_t)(l1 - l0) * H * D * tokens;",
                        "return (int64_t)(l1 - l0) * H * D * tokens;"),
    # the sampled lookup one element off inside a token
    "source_of_d_shifted": ("t = seq_start[b] + r / D, d = r % D;",
                            "t = seq_start[b] + r / D, d = (r + 1) % D;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = (Path(oracle.__file__).parent / "dv_oracle.c").read_text()
    old, new = MUTANTS[name]
    assert old in src, name
    mutated = src.replace(old, new)
    if name == "d_reversed":  # copy d in reverse order inside each token
        mutated = mutated.replace("P * k_index(layer_stride, B, H, D, S, x, l, b, h, t, d)",
                                  "P * k_index(layer_stride, B, H, D, S, x, l, b, h, t, dflip - d)")
    cpath = tmp_path / "mutant.c"
    cpath.write_text(mutated)
    lib = oracle.build(cpath, tmp_path / "libmutant.so")
    r = subprocess.run([sys.executable, str(Path(P.__file__)), str(lib)],
                       cwd=str(Path(P.__file__).parent.parent), capture_output=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin"


def test_restore_overlapping_records_later_wins():
    """Records unpacked in append order: where a later record covers slices an
    earlier one wrote, the later bytes stay (the replica log of Fig 10 is
    replayed in order).  Expected cache built from the independent layout
    masks alone: B's bytes where B selects, else A's where A selects, else 0."""
    g = Geometry("o", 3, 3, 2, 32, 16, 2, "raw")
    rng = np.random.default_rng(24)
    ka, va = P.random_cache(g, rng)
    kb, vb = P.random_cache(g, rng)
    sa, ea = np.array([0, 2, 5], np.int32), np.array([9, 7, 16], np.int32)
    sb, eb = np.array([4, 0, 15], np.int32), np.array([12, 3, 16], np.int32)
    recs = [(0, 3, sa, ea, ORC.pack(g, ka, va, 0, 3, sa, ea)),
            (1, 3, sb, eb, ORC.pack(g, kb, vb, 1, 3, sb, eb))]
    k2, v2 = ORC.restore(g, recs)
    mka, mva = (np.repeat(m, 2) for m in P.selected_mask(g, 0, 3, sa, ea))
    mkb, mvb = (np.repeat(m, 2) for m in P.selected_mask(g, 1, 3, sb, eb))
    assert (mka & mkb).any()  # the records do overlap
    want_k = np.where(mkb, kb, np.where(mka, ka, 0)).astype(np.uint8)
    want_v = np.where(mvb, vb, np.where(mva, va, 0)).astype(np.uint8)
    assert np.array_equal(k2, want_k) and np.array_equal(v2, want_v)
