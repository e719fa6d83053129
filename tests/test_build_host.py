"""The build's staleness check: a library counts as up to date only for the flags it
was built with (CPU, no compiler run)."""
import os

from block_quantized_wire_gb300 import build


def test_flag_stamp_decides_staleness(tmp_path):
    lib = str(tmp_path / "libbq_test.so")
    with open(lib, "wb") as f:
        f.write(b"\0")
    assert not build.up_to_date(lib)  # no stamp: rebuild
    with open(lib + ".flags", "w") as f:
        f.write(build._flag_stamp(["-DBQ_HOP_WIDE=0"]))
    newer = max(os.path.getmtime(p) for p in build._inputs()) + 10
    os.utime(lib, (newer, newer))
    assert build.up_to_date(lib, ["-DBQ_HOP_WIDE=0"])
    assert not build.up_to_date(lib)  # built with other flags than the default
    assert not build.up_to_date(lib, ["-DBQ_HOP_WIDE=1"])
    os.utime(lib, (newer - 1e6, newer - 1e6))
    assert not build.up_to_date(lib, ["-DBQ_HOP_WIDE=0"])  # older than a source
