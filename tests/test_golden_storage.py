"""Storage of the packed codes against the figures the method pages print (tests/golden).

Host-only: kvq_page_layout is arithmetic on the configuration, so these run without a GPU."""
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_cache_storage.txt")


@pytest.fixture(scope="module")
def kvq():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    from bit_asymmetric_kv_kvq_gb300 import _build
    try:
        _build.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    return kvq


def golden():
    rows, scalars = {}, {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split(":", 1)
        vals = [float(x) for x in val.split()]
        if len(vals) == 1:
            scalars[key] = vals[0]
        else:
            rows[key] = vals
    return rows, scalars


def code_bytes(kvq, k_bits, v_bits, R=128, G=32):
    """Bytes of one page's key and value code sections (tokens_per_page tokens, D = 128)."""
    lay = kvq.kvq_page_layout(kvq.make_config(1, 1, 1, 128, 4096, k_bits, v_bits, G, R))
    return lay["kmeta_offset"] - lay["kcodes_offset"], lay["vmeta_offset"] - lay["vcodes_offset"], lay


def test_fixture_is_complete():
    rows, scalars = golden()
    assert set(rows) == {"LLaMA-7B", "LLaMA-13B", "LLaMA-30B", "LLaMA-65B"}
    assert all(len(v) == 4 for v in rows.values())
    assert set(scalars) == {"k4v2_saving_vs_k4v4", "k4v2_value_share_vs_k4v4"}


@pytest.mark.parametrize("R,G", [(128, 32), (128, 64), (64, 32), (32, 32)])
def test_code_sections_cost_the_printed_fraction_of_fp16(kvq, R, G):
    """int4 / int3 / int2 rows of the KVQuant review's table: B/16 of the fp16 baseline, to the
    printed digit, whatever the page shape (3-bit codes packed densely, no padding waste)."""
    rows, _ = golden()
    for model, (base, *printed) in rows.items():
        for bits, want in zip((4, 3, 2), printed):
            kb, vb, lay = code_bytes(kvq, bits, bits, R, G)
            fp16 = 2 * (2 * lay["tokens_per_page"] * 128)  # the same tokens' keys and values in fp16
            ours = base * (kb + vb) / fp16
            assert abs(ours - want) <= 0.05 + 1e-9, (model, bits, ours, want)


def test_k4v2_against_k4v4(kvq):
    """The mixed-width page: a quarter of the code bytes saved, the values' half of theirs."""
    _, scalars = golden()
    kb42, vb42, _ = code_bytes(kvq, 4, 2)
    kb44, vb44, _ = code_bytes(kvq, 4, 4)
    assert kb42 == kb44
    assert 1.0 - (kb42 + vb42) / (kb44 + vb44) == pytest.approx(scalars["k4v2_saving_vs_k4v4"])
    assert vb42 / vb44 == pytest.approx(scalars["k4v2_value_share_vs_k4v4"])
