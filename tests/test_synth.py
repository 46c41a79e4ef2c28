"""The seeded input generator against its published definition (CPU)."""
import numpy as np

import synth
from synth import configs
from tests.oracle_pins import read_golden


def test_splitmix64_published_vectors():
    gd = read_golden("splitmix64_seed1234567.txt")
    want = [int(t) for t in gd["outputs"].split()]
    got = [int(t) for t in synth.splitmix64_sequence(int(gd["seed"]), len(want))]
    assert got == want


def test_fill_word_n_is_output_n():
    base = synth.stream_base(99, 1)
    words = synth.fill_bytes(99, 1, 8 * 64, "raw").view("<u8")
    assert np.array_equal(words, synth.splitmix64_sequence(base, 64))


def test_fill_is_finite_for_float_kinds():
    for kind, dt in (("fp16", np.float16), ("fp32", np.float32)):
        vals = synth.fill_bytes(5, 0, 1 << 20, kind).view(dt)
        assert np.isfinite(vals).all()
    bf = synth.fill_bytes(5, 0, 1 << 20, "bf16").view(np.uint16)
    assert not ((bf & 0x7F80) == 0x7F80).any()
    raw = synth.fill_bytes(5, 0, 1 << 20, "raw").view(np.uint16)
    assert ((raw & 0x7C00) == 0x7C00).any()  # raw keeps what was drawn


def test_fill_elements_matches_fill_bytes():
    rng = np.random.default_rng(1)
    for eb, kind in ((2, "fp16"), (2, "bf16"), (4, "fp32"), (1, "raw")):
        full = synth.fill_bytes(17, 1, 4096, kind)
        dt = {1: np.uint8, 2: np.uint16, 4: np.uint32}[eb]
        idx = rng.integers(0, 4096 // eb, size=200)
        assert np.array_equal(synth.fill_elements(17, 1, idx, eb, kind), full.view(dt)[idx])


def test_k_and_v_streams_differ():
    a = synth.fill_bytes(3, 0, 1024, "raw")
    b = synth.fill_bytes(3, 1, 1024, "raw")
    assert not np.array_equal(a, b)


def test_workload_draws_are_seeded_and_in_range():
    l3 = configs.opt13b_lengths()
    assert np.array_equal(l3, configs.opt13b_lengths())
    assert l3.min() >= 16 and l3.max() <= 2048 and l3.size == 8
    for p, o in configs.opt66b_microbatches():
        assert p.min() >= 16 and p.max() <= 1024
        assert o.min() >= 1 and (p + o).max() <= 2047
    l5 = configs.bloom_lengths()
    assert l5.min() >= 64 and l5.max() <= 1536
    assert (l5 + configs.BLOOM_DECODE_STEPS).max() <= configs.BLOOM_STAGE.max_seq


def test_fill_bytes_offset_and_threads_give_the_same_bytes():
    """A window [offset, offset + n) of the fill equals that slice of the whole
    fill, and the threaded fill equals the serial one."""
    for kind in ("fp16", "bf16", "raw"):
        whole = synth.fill_bytes(11, 0, 1 << 22, kind)
        for off, n in ((0, 4096), (8, 800), (1 << 20, 1 << 20), ((1 << 22) - 64, 64)):
            assert np.array_equal(synth.fill_bytes(11, 0, n, kind, offset=off), whole[off:off + n])
        big = synth.fill_bytes(12, 1, 3 << 25, kind, offset=1 << 21)
        assert np.array_equal(synth.fill_bytes(12, 1, 3 << 25, kind, offset=1 << 21, threads=4), big)
