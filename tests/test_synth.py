"""The seeded generators: published splitmix64 outputs, determinism, and the
value ranges of each synthetic workload's fields."""

import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_reference_outputs():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "splitmix64_seed0.txt"))
            if ln.strip() and not ln.startswith("#")]
    z = synth.Stream(0).draw(len(rows))
    for (i, hexv), v in zip(rows, z):
        assert int(v) == int(hexv, 16)


def test_stream_is_counter_based():
    a = synth.Stream(42).draw(10)
    st = synth.Stream(42)
    b = np.concatenate([st.draw(3), st.draw(7)])
    assert np.array_equal(a, b)


def test_q4k_fields_in_range():
    w = synth.gen_q4k_rows(synth.Stream(0), 64, 512).reshape(-1, 144)
    d = w[:, 0:2].copy().view(np.float16).astype(np.float64).ravel()
    dmin = w[:, 2:4].copy().view(np.float16).astype(np.float64).ravel()
    assert d.min() >= 1e-3 * (1 - 2 ** -10) and d.max() <= 4e-3 * (1 + 2 ** -10)
    assert dmin.min() >= 0 and dmin.max() <= 2e-3 * (1 + 2 ** -10)


def test_q6k_and_q8_0_fields_in_range():
    w6 = synth.gen_q6k_rows(synth.Stream(4), 32, 512).reshape(-1, 210)
    sc = w6[:, 192:208].view(np.int8)
    assert sc.min() == -64 and sc.max() == 63
    d6 = w6[:, 208:210].copy().view(np.float16).astype(np.float64)
    assert d6.min() >= 1e-4 * (1 - 2 ** -10) and d6.max() <= 5e-4 * (1 + 2 ** -10)
    w8 = synth.gen_q8_0_rows(synth.Stream(2), 64, 1024).reshape(-1, 34)
    q = w8[:, 2:].view(np.int8)
    assert q.min() == -127 and q.max() == 127


def test_moe_ids_distinct_and_normal_moments():
    ids = synth.gen_moe_ids(synth.Stream(3), 8, 128)
    assert len(set(ids.tolist())) == 8 and ids.min() >= 0 and ids.max() < 128
    x = synth.gen_normal(synth.Stream(1), 200000)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1) < 0.01


def test_config_shapes():
    c = synth.make_config("q4k_256x1024")
    assert c["w"].shape == (256, 576) and c["x"].shape == (1024,)
    assert synth.row_bytes("q6k", 14336) == 11760 and synth.row_bytes("q8_0", 4096) == 4352
