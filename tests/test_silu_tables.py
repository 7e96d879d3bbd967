"""The GPU kernels' silu tables (fp8_token_group_gb300/csrc/silu_tables.inc) are generated
data.  Regenerating them re-runs the generator's own checks: the closed forms outside each
table (S = g/2, g or -0 for bf16; S = g or -0 for fp16) for every 16-bit gate of both types.
The committed file must then match the regenerated one byte for byte.  CPU only; no kernel
runs."""
import importlib.util
import os

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "fp8_token_group_gb300", "csrc")


def test_committed_silu_tables_regenerate_identically(tmp_path):
    pytest.importorskip("mpmath")
    spec = importlib.util.spec_from_file_location("gen_silu_tables",
                                                  os.path.join(CSRC, "gen_silu_tables.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    out = tmp_path / "silu_tables.inc"
    gen.main(str(out))                       # raises if any generator check fails
    with open(os.path.join(CSRC, "silu_tables.inc")) as f:
        committed = f.read()
    assert out.read_text() == committed
