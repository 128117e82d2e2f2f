"""CPU checks of the C ABI: the library loads, exports every entry point that
include/kvq.h declares, and its host-only functions agree with the oracle."""
import os
import re

import pytest

from conftest import ROOT


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("kvq_create_cache", "kvq_destroy_cache", "kvq_quantize_and_store",
              "kvq_decode_attention", "kvq_decode_workspace_size", "kvq_dequantize",
              "kvq_cache_layout", "kvq_bytes_per_token", "kvq_format_from_name",
              "kvq_format_name", "kvq_get_device_error", "kvq_last_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(kvq):
    for n in _declared():
        assert hasattr(kvq.lib, n), n


def test_format_names_round_trip(kvq):
    for name, code in kvq.FORMATS.items():
        assert kvq.kvq_format_name(code) == name
        assert kvq.kvq_format_from_name(name) == code
    assert kvq.kvq_format_name(99) is None
    with pytest.raises(kvq.KVQError):
        kvq.kvq_format_from_name("fp8")


@pytest.mark.parametrize("fmt", ["bf16", "fp8_e4m3", "fp8_e5m2", "fp4_mx_block16", "nvfp4"])
def test_bytes_per_token_matches_oracle(kvq, orc, fmt):
    for L, H, D in ((80, 8, 128), (32, 8, 128), (1, 1, 16), (61, 1, 576)):
        assert kvq.kvq_bytes_per_token(fmt, L, H, D) == orc.bytes_per_token(fmt, L, H, D)
    assert kvq.kvq_bytes_per_token(fmt, 1, 1, 24) == 0   # head_dim % 16 != 0


def test_create_cache_rejects_bad_arguments_before_device_work(kvq):
    for args in (("fp8_e4m3", 1, 8, 120, 16, 4), ("fp8_e4m3", 0, 8, 128, 16, 4),
                 (7, 1, 8, 128, 16, 4), ("nvfp4", 1, 8, 128, 0, 4)):
        with pytest.raises(kvq.KVQError) as e:
            kvq.kvq_create_cache(*args)
        assert e.value.code == "KVQ_ERR_INVALID_ARG"


def test_noalloc_null_cache_is_an_invalid_argument(kvq):
    """The allocation-free decode entry point reports a NULL cache as
    KVQ_ERR_INVALID_ARG before touching the device (no GPU needed)."""
    st = kvq.lib.kvq_decode_attention_noalloc(None, 0, None, 64, None, 4, None, 2, 0.1, None, None)
    assert kvq._binding._STATUS[st] == "KVQ_ERR_INVALID_ARG"
    assert "NULL" in kvq.kvq_last_error_string()
