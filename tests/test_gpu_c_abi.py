"""The C ABI from a plain C99 program on the GPU: tests/c/transfer_from_c.c moves a request
between two pools through kvx_transfer, checks every destination byte against the definition
of the move, and checks that a request with a slot past the end moves nothing."""
import subprocess

import pytest

from tests.cprog import build_c_program

pytestmark = pytest.mark.gpu


def test_transfer_from_c(tmp_path):
    torch = pytest.importorskip("torch")
    assert torch.cuda.is_available()
    exe = build_c_program(str(tmp_path / "transfer_from_c"))
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.strip() == "ok"
