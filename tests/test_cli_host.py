"""Host-only parsing of the command-line tool's explicit configuration."""
import pytest

from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.cli import parse_cfg


def test_parse_cfg_fields():
    c = parse_cfg("kind=cc,split_k=2,block=128,rows=4,k_unroll=1")
    d = c.as_dict()
    assert d["kind"] == "cc" and d["split_k"] == 2 and d["block"] == 128
    assert d["rows"] == 4 and d["k_unroll"] == 1 and d["flags"] == binding.FLAG_PDL


def test_parse_cfg_defaults_and_flags():
    d = parse_cfg("kind=tc05,split_k=8,flags=3").as_dict()
    assert d["kind"] == "tc05" and d["split_k"] == 8 and d["flags"] == 3


@pytest.mark.parametrize("text", ["split_k=2", "kind=cc,bogus=1", "kind=cc,split_k=", "kind=cc,split_k=x"])
def test_parse_cfg_rejects(text):
    with pytest.raises(ValueError):
        parse_cfg(text)
