"""Wire-mode selection by name, on CPU ("feat(pcie_dma): add INT8 and MXFP8 wire modes",
Modes: whitespace and case are normalized, an unknown non-empty name raises instead of
silently selecting another mode, an empty name keeps the BF16 path)."""
import pytest

from block_quantized_wire_gb300 import topology


@pytest.mark.parametrize("name", sorted(topology.MODES))
def test_every_mode_name_selects_its_topology(name):
    assert topology.select_mode(name) is topology.MODES[name]
    assert topology.select_mode(f"  {name.upper()}\t") is topology.MODES[name]
    assert topology.select_mode(name.title()) is topology.MODES[name]


def test_page_mode_names_are_all_accepted():
    for name in ("i8", "i8_ring", "i8_a2a", "mx", "mx_ring", "mx_a2a"):
        assert topology.select_mode(name) is not None


@pytest.mark.parametrize("empty", [None, "", "   ", "\n"])
def test_empty_name_keeps_the_bf16_path(empty):
    assert topology.select_mode(empty) is None


@pytest.mark.parametrize("typo", ["mx_rnig", "i8ring", "i8-ring", "int8", "mxfp8", "e4m3", "i8_a2a_"])
def test_unknown_names_raise(typo):
    with pytest.raises(ValueError):
        topology.select_mode(typo)
