"""Usage-history files in the route_trace format, on the host (no GPU): the
writer against the format's rules (colibri tuning guide, gitcode.com,
"usage-history format") and a hand-written example, the engine id against the
value the guide prints, and the reader's refusals."""
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GLM_ID = 3815245270          # the guide's FNV-1a value for "glm_moe_dsa"


@pytest.fixture(scope="module")
def moe():
    import expert_routing_grouped_gb300 as m
    return m


def load_example():
    engine, counts, expect = None, [], []
    for line in open(os.path.join(ROOT, "tests", "golden", "route_trace_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        key, rest = line.split(" ", 1)
        if key == "engine":
            engine = rest.strip()
        elif key == "counts":
            counts.append([int(v) for v in rest.split()])
        elif key == "expect":
            expect.append(rest.strip())
    return engine, np.array(counts, np.int64), expect


def test_engine_id_matches_the_guide(moe):
    assert moe.engine_id("glm_moe_dsa") == GLM_ID
    assert GLM_ID > 2**31 - 1                      # why the id sits in the third field
    assert moe.engine_id("") == 2166136261        # FNV-1a of nothing is the offset basis
    # one byte: (basis xor byte) * prime mod 2^32
    assert moe.engine_id("a") == ((2166136261 ^ 0x61) * 16777619) % 2**32
    assert moe.engine_id("kimi_k3") != GLM_ID
    assert moe.lib.moe_engine_id(None) == 0


def test_writer_matches_the_example(moe, tmp_path):
    engine, counts, expect = load_example()
    p = tmp_path / "usage"
    moe.route_trace_write(p, counts, engine)
    data = p.read_bytes()
    assert data == ("\n".join(expect) + "\n").encode()


def test_every_record_has_three_integer_fields(moe, tmp_path):
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 5, (6, 64)) * (rng.random((6, 64)) < 0.3)
    counts[2, 5] = 2**40                            # counts are 64-bit
    p = tmp_path / "usage"
    moe.route_trace_write(p, counts, "glm_moe_dsa")
    lines = p.read_text().splitlines()
    assert lines[0] == "-1 6 64" and lines[1] == "-2 1 %d" % GLM_ID
    data = lines[2:]
    assert len(data) == np.count_nonzero(counts)    # sparse: non-zero counts only
    prev = (-1, -1)
    for ln in lines:
        f = ln.split(" ")
        assert len(f) == 3 and all(v.lstrip("-").isdigit() for v in f)
    for ln in data:
        l, e, c = map(int, ln.split())
        assert (l, e) > prev and c == counts[l, e] and c > 0    # layer-major, ascending
        prev = (l, e)


def test_round_trip(moe, tmp_path):
    rng = np.random.default_rng(11)
    counts = rng.integers(0, 1000, (3, 256)) * (rng.random((3, 256)) < 0.1)
    p = tmp_path / "usage"
    moe.route_trace_write(p, counts, "glm_moe_dsa")
    back, found = moe.route_trace_read(p, 3, 256, "glm_moe_dsa")
    assert found == GLM_ID
    assert np.array_equal(back, counts)


def test_empty_history_is_a_zero_byte_file(moe, tmp_path):
    p = tmp_path / "usage"
    p.write_text("stale\n")
    moe.route_trace_write(p, np.zeros((4, 8), np.int64), "glm_moe_dsa")
    assert p.stat().st_size == 0
    back, found = moe.route_trace_read(p, 4, 8, "glm_moe_dsa")
    assert found == 0 and not back.any()


def test_reader_refuses_another_engine(moe, tmp_path):
    p = tmp_path / "usage"
    counts = np.zeros((2, 4), np.int64)
    counts[1, 2] = 5
    moe.route_trace_write(p, counts, "kimi_k3")
    with pytest.raises(moe.MoeError) as e:
        moe.route_trace_read(p, 2, 4, "glm_moe_dsa")
    assert e.value.code == moe.MOE_ERR_ENGINE
    # an explicitly trusted file (engine 0) is read whoever wrote it
    back, found = moe.route_trace_read(p, 2, 4, 0)
    assert found == moe.engine_id("kimi_k3") and back[1, 2] == 5
    # the dimensions are checked either way
    with pytest.raises(moe.MoeError) as e:
        moe.route_trace_read(p, 2, 8, 0)
    assert e.value.code == moe.MOE_ERR_ENGINE


def test_reader_adds_and_leaves_counts_alone_on_error(moe, tmp_path):
    import ctypes
    p = tmp_path / "usage"
    c = np.zeros((1, 4), np.int64)
    c[0, 1] = 2
    moe.route_trace_write(p, c, "glm_moe_dsa")
    acc = np.full((1, 4), 10, np.int64)
    rc = moe.lib.moe_route_trace_read(os.fsencode(p), 1, 4, GLM_ID, acc.ctypes.data, None)
    assert rc == 0 and acc.tolist() == [[10, 12, 10, 10]]
    rc = moe.lib.moe_route_trace_read(os.fsencode(p), 1, 4, 12345, acc.ctypes.data, None)
    assert rc == moe.MOE_ERR_ENGINE and acc.tolist() == [[10, 12, 10, 10]]
    bad = tmp_path / "bad"
    bad.write_text("-1 1 4\n0 1 3\n0 2\n")
    rc = moe.lib.moe_route_trace_read(os.fsencode(bad), 1, 4, 0, acc.ctypes.data, None)
    assert rc == moe.MOE_ERR_IO and acc.tolist() == [[10, 12, 10, 10]]
    assert moe.lib.moe_route_trace_read(os.fsencode(tmp_path / "missing"), 1, 4, 0,
                                        acc.ctypes.data, ctypes.c_void_p()) == moe.MOE_ERR_IO


def test_reader_skips_unknown_headers_and_takes_headerless_files(moe, tmp_path):
    p = tmp_path / "usage"
    p.write_text("-1 2 4\n-3 7 9\n-2 1 %d\n1 3 4\n\n0 0 1\n1 3 2\n" % GLM_ID)
    back, found = moe.route_trace_read(p, 2, 4, "glm_moe_dsa")
    assert found == GLM_ID
    assert back.tolist() == [[1, 0, 0, 0], [0, 0, 0, 6]]
    p.write_text("0 2 5\r\n1 1 1\r\n")                # the older form: triplets only
    back, found = moe.route_trace_read(p, 2, 4, "glm_moe_dsa")
    assert found == 0 and back.tolist() == [[0, 0, 5, 0], [0, 1, 0, 0]]


@pytest.mark.parametrize("text", [
    "0 1 2 3\n",                     # four fields would throw a scanf reader out of step
    "0 1\n",
    "glm 1 2\n",                     # no string fields
    "-2 1 glm_moe_dsa\n",
    "0 1 2x\n",
    "2 0 1\n",                       # layer out of range
    "0 4 1\n",                       # expert out of range
    "0 1 -3\n",                      # negative count
    "-2 1 4294967296\n",             # an engine id wider than 32 bits
])
def test_reader_rejects_malformed_records(moe, tmp_path, text):
    p = tmp_path / "usage"
    p.write_text(text)
    with pytest.raises(moe.MoeError) as e:
        moe.route_trace_read(p, 2, 4, 0)
    assert e.value.code == moe.MOE_ERR_IO


def test_writer_rejects_bad_arguments(moe, tmp_path):
    p = os.fsencode(tmp_path / "usage")
    c = np.zeros((1, 4), np.int64)
    c[0, 0] = -1
    assert moe.lib.moe_route_trace_write(p, 1, 4, 0, c.ctypes.data) == moe.MOE_ERR_ARG
    assert moe.lib.moe_route_trace_write(p, 0, 4, 0, c.ctypes.data) == moe.MOE_ERR_ARG
    assert moe.lib.moe_route_trace_write(None, 1, 4, 0, c.ctypes.data) == moe.MOE_ERR_ARG
    assert moe.lib.moe_route_trace_write(os.fsencode(tmp_path / "no" / "dir"), 1, 4, 0,
                                         np.ones(4, np.int64).ctypes.data) == moe.MOE_ERR_IO
