"""The bench's end-to-end leg reads back what the steps computed (GPU).

With the copies overlapped (double-buffered gradients, parameters read back
from a device snapshot during the next step), the parameters that reach the
host after the last step must be bitwise those of the same steps run with
the copies in line, and those left on the device.
"""
import pytest
import torch

import bench
import workloads
from matrix_orthogonalising_optimizer_gb300 import Muon


@pytest.mark.gpu
def test_overlapped_copies_read_back_the_final_parameters():
    cfg = workloads.get("c2")
    shapes = [(r, c, 0) for r, c in cfg.shapes]
    stream = torch.cuda.current_stream()
    results = {}
    for overlap in (False, True):
        muon = Muon(shapes).bind()
        ws, gs, ms = workloads.make_set(cfg, "cuda")
        host = []
        out = bench.measure_e2e(muon, cfg, ws, gs, ms, 3, stream, 1, overlap=overlap, host_out=host)
        torch.cuda.synchronize()
        assert out["h2d_bytes_per_step"] == sum(g.numel() * 2 for g in gs)
        assert ("overlapped" in out["copies"]) == overlap
        assert muon.device_status() == 0
        for h, w in zip(host, ws):
            assert torch.equal(h, w.cpu())
        results[overlap] = host
    for a, b in zip(results[False], results[True]):
        assert torch.equal(a, b)
