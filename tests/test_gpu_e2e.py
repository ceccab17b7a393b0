"""The end-to-end measurement's pipeline returns the op's results: each row
block copied in from pinned host memory, run through the op and copied back
(graph-replayed and eager) must equal a direct call of the op on that block's
rows in device memory, byte for byte (same rows, same launch shape).  Covers
a ragged last block, NVFP4 scales split at 128-row tiles (the last block
taking the padding rows), y, no residual and k partials (one block)."""
import dataclasses

import pytest
import torch

import bench
from nvfp4_quant_gemma_gb300.workloads import all_workloads, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gnq():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from nvfp4_quant_gemma_gb300 import build
    build.build()
    import nvfp4_quant_gemma_gb300 as pkg
    pkg.load()
    pkg.set_launch_policy(0, 0, 0, 0)
    pkg.set_pdl(True)
    return pkg


def _small(name, M, H, **kw):
    return dataclasses.replace(all_workloads()[name], M=M, H=H, name=f"{name}_{M}x{H}", **kw)


CASES = [
    _small("prefill_m16384_h8192_fp16_fp8", 1000, 2048),
    _small("prefill_m2048_h5120_bf16_nvfp4_y", 300, 1024),
    _small("prefill_m16384_h8192_fp16_nvfp4_nores", 640, 4096),
    _small("prefill_m16384_h8192_fp16_mxfp8", 200, 1024),
    _small("parts4_m4096_h7168_bf16_nvfp4_y", 256, 1024),
]


def _direct(gnq, wl, inp, dev, a, e):
    """The op on rows [a, e) in device memory, outputs allocated for that block."""
    w, s = inp["weight"].to(dev), inp["scale"].to(dev)
    if wl.k > 1:
        x = inp["x"][:, a:e].contiguous().to(dev)
    else:
        x = inp["x"][a:e].contiguous().to(dev)
    r = None if inp["residual"] is None else inp["residual"][a:e].contiguous().to(dev)
    out = gnq.alloc_outputs(e - a, wl.H, wl.mode, wl.write_y, x)
    if wl.k > 1:
        gnq.gemma_add_rms_norm_quant_parts(x, r, w, wl.eps, s, wl.mode, write_y=wl.write_y, out=out)
    else:
        gnq.gemma_add_rms_norm_quant(x, r, w, wl.eps, s, wl.mode, write_y=wl.write_y, out=out)
    torch.cuda.synchronize(dev)
    return out, r


def _u8(t):
    return t.contiguous().view(torch.uint8).cpu()


@pytest.mark.parametrize("graph", [True, False], ids=["graph", "eager"])
@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
def test_pipeline_returns_the_op_results(gnq, wl, graph):
    dev = torch.device("cuda")
    chunks = 4
    res = []
    bench.e2e_measure(gnq, wl, dev, steps=5, warmup=2, graph=graph, chunks=chunks, results=res)
    assert len(res) == 2
    inp = make_inputs(wl)
    blocks = bench.row_blocks(wl.M, chunks if wl.k == 1 else 1)
    assert len(blocks) == 1 if wl.k > 1 else 1 < len(blocks) <= chunks
    for (q_h, bs_h, y_h), r_h in res:
        for a, e in blocks:
            (q, bs, y), r = _direct(gnq, wl, inp, dev, a, e)
            assert torch.equal(_u8(q_h[a:e]), _u8(q))
            if wl.mode == "nvfp4":
                # the block's 128-row tiles; only rows a..e-1 of them are defined
                tiles = _u8(bs_h[a:a + bs.shape[0]]).reshape(-1, 128, bs.shape[1])
                want = _u8(bs).reshape(-1, 128, bs.shape[1])
                wp = bs.shape[1]
                for ti in range(want.shape[0]):
                    n = min(128, e - a - 128 * ti)
                    # swizzled 128x4 tiles: row rr's four scales of column
                    # tile ct sit at ct * 512 + (rr % 32) * 16 + (rr // 32) * 4
                    idx = torch.tensor([ct * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc
                                        for rr in range(n) for ct in range(wp // 4)
                                        for cc in range(4)])
                    assert torch.equal(tiles[ti].reshape(-1)[idx], want[ti].reshape(-1)[idx])
            elif wl.mode == "mxfp8":
                assert torch.equal(_u8(bs_h[a:e]), _u8(bs))
            if wl.write_y:
                assert torch.equal(_u8(y_h[a:e]), _u8(y))
            if r is not None:
                assert torch.equal(_u8(r_h[a:e]), _u8(r))
    assert gnq.read_device_error() == 0
