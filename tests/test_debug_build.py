"""The debug build (device-side index checks that write DF_EINVAL to the status word and skip
the access): it compiles for sm_103a and exports the same symbols (CPU), and a draft round run
with it matches the CPU oracle with a clean status word (GPU)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _debug_lib():
    from speculative_decoding_drafter_dflash_gb300 import build
    return build.build(debug=True)


def test_debug_build_compiles_and_exports_the_abi():
    import ctypes
    path = _debug_lib()
    assert os.path.exists(path)
    L = ctypes.CDLL(path)
    from speculative_decoding_drafter_dflash_gb300 import binding
    for name, _, _ in binding._SIGS:
        assert hasattr(L, name), name


@pytest.mark.gpu
def test_debug_build_round_matches_oracle():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = _debug_lib()
    env = dict(os.environ, DFLASH_LIB=path)
    r = subprocess.run([sys.executable, "-c", "import __graft_entry__ as g; g.smoke()"], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "smoke ok" in r.stdout
