"""The tensor-core plumbing the attention kernels rely on, one tile at a time:
128-byte-swizzled TMA tiles, K-major and MN-major shared-memory descriptors,
the instruction descriptor and A operands in TMEM, against a CPU product."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [128, 64])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_umma_tile_matches_cpu_product(cuda_device, mode, n):
    import tiled_scaled_dot_gb300 as g
    a = synth.normal((128, 128), 5, 0, torch.bfloat16)
    b = synth.normal((n, 128) if mode == 0 else (128, n), 5, 1, torch.bfloat16)
    ref = a.double() @ (b.double().T if mode == 0 else b.double())
    c = g.diag_umma(mode, a.to(cuda_device), b.to(cuda_device), n)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    err = (c.double().cpu() - ref).abs().max().item()
    assert err < 1e-3, f"mode {mode} n {n}: max err {err}"


def test_bounded_wait_runs_out_and_reports(cuda_device):
    """The failure path of the bounded waits, without a fault: a wait that
    nothing satisfies gives up after its limit, records its site in the device
    status word, and leaves the context usable."""
    import tiled_scaled_dot_gb300 as g
    g.device_status()  # start clear
    g.diag_wait_timeout(20_000_000)  # 20 ms
    st = g.device_status(clear=False)
    assert st & (1 << 16), f"status {st:#x}"
    assert g.device_status() == st  # read and clear
    assert g.device_status() == 0
    # the context still runs tensor-core work correctly
    a = synth.normal((128, 128), 6, 0, torch.bfloat16)
    b = synth.normal((128, 128), 6, 1, torch.bfloat16)
    c = g.diag_umma(0, a.to(cuda_device), b.to(cuda_device), 128)
    assert g.device_status() == 0
    assert (c.double().cpu() - a.double() @ b.double().T).abs().max().item() < 1e-3
