"""The hardware-rate probes behind the kernels' design choices
(`bench.py --probe ...`) compile for sm_103a (no GPU needed)."""
import os
import shutil

import pytest

from mla_decode_context_gb300 import build_lib


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="no nvcc")
@pytest.mark.parametrize("name", build_lib.PROBES)
def test_probe_compiles(name):
    exe = build_lib.build_probe(name)
    assert os.path.isfile(exe) and os.access(exe, os.X_OK)
