"""The compute-free stream probes behind the benchmark's ceiling figures
(libmpprobe.so) must move exactly the step's bytes, or their throughput
means nothing: master, m and v come back unchanged and the weight receives
the gradient's bits, through register loads and through TMA bulk copies;
the bulk copy probe copies its tiles exactly. No probe wait may give up."""
import ctypes
import os
import time

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TILE = 2048


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    lib = ctypes.CDLL(os.path.join(ROOT, "mixed_precision_adamw_gb300", "libmpprobe.so"))
    vp, u64, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int
    lib.mp_probe_step_streams.argtypes = [vp, vp, vp, vp, vp, u64, i32, vp]
    lib.mp_probe_step_streams_bulk.argtypes = [vp, vp, vp, vp, vp, u64, i32, i32, i32, vp, vp]
    lib.mp_probe_step_streams_bulk_tile.argtypes = [vp, vp, vp, vp, vp, u64, ctypes.c_uint32, i32, i32, i32, vp, vp]
    lib.mp_probe_copy_bulk.argtypes = [vp, vp, u64, i32, i32, i32, vp, vp]
    lib.mp_probe_bulk_timeout.argtypes = [vp, u64, vp, vp]
    return lib


def _streams(n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    grads = torch.randint(-32768, 32767, (n,), generator=g, device="cuda", dtype=torch.int16)
    master, m, v = (torch.randn(n, generator=g, device="cuda") for _ in range(3))
    params = torch.zeros(n, dtype=torch.int16, device="cuda")
    return params, grads, master, m, v


@pytest.mark.parametrize("kind,bps,stages,hint", [("reg", 3, 0, 0), ("reg", 8, 0, 0), ("bulk", 1, 7, 1),
                                                  ("bulk", 1, 2, 0), ("bulk", 2, 3, 1)])
@pytest.mark.parametrize("tiles", [5, 600, 4999])
def test_step_stream_probes_move_the_step_bytes(probe, kind, bps, stages, hint, tiles):
    n = tiles * TILE
    params, grads, master, m, v = _streams(n, tiles)
    keep = [x.clone() for x in (master, m, v)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if kind == "reg":
        rc = probe.mp_probe_step_streams(params.data_ptr(), grads.data_ptr(), master.data_ptr(), m.data_ptr(),
                                         v.data_ptr(), n, bps, s)
    else:
        rc = probe.mp_probe_step_streams_bulk(params.data_ptr(), grads.data_ptr(), master.data_ptr(),
                                              m.data_ptr(), v.data_ptr(), n, bps, stages, hint, err.data_ptr(), s)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(params, grads)
    for a, b in zip((master, m, v), keep):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("tile,stages", [(64, 8), (2304, 3), (6144, 2), (8192, 2)])
@pytest.mark.parametrize("tiles", [3, 601])
def test_step_stream_probe_with_other_tile_sizes_moves_the_step_bytes(probe, tile, stages, tiles):
    n = tiles * tile
    params, grads, master, m, v = _streams(n, tiles + tile)
    keep = [x.clone() for x in (master, m, v)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.mp_probe_step_streams_bulk_tile(params.data_ptr(), grads.data_ptr(), master.data_ptr(), m.data_ptr(),
                                               v.data_ptr(), n, tile, 1, stages, 1, err.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(params, grads)
    for a, b in zip((master, m, v), keep):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("bps,stages,hint", [(1, 7, 1), (2, 3, 0)])
def test_bulk_copy_probe_copies_its_tiles(probe, bps, stages, hint):
    tile_bytes = TILE * 14
    tiles = 3001
    src = torch.randint(0, 255, (tiles * tile_bytes + 4096,), dtype=torch.uint8, device="cuda")
    dst = torch.zeros_like(src)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.mp_probe_copy_bulk(dst.data_ptr(), src.data_ptr(), tiles, bps, stages, hint, err.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(dst[: tiles * tile_bytes], src[: tiles * tile_bytes])
    assert int(dst[tiles * tile_bytes:].count_nonzero()) == 0  # nothing past the last tile


def test_bulk_probe_refuses_bad_arguments(probe):
    n = 4 * TILE
    params, grads, master, m, v = _streams(n, 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (params.data_ptr(), grads.data_ptr(), master.data_ptr(), m.data_ptr(), v.data_ptr())
    assert probe.mp_probe_step_streams_bulk(*args, n + 1, 1, 4, 0, err.data_ptr(), s) != 0  # not whole tiles
    assert probe.mp_probe_step_streams_bulk(*args, n, 1, 1, 0, err.data_ptr(), s) != 0  # one stage
    assert probe.mp_probe_step_streams_bulk(*args, n, 1, 9, 0, err.data_ptr(), s) != 0  # too many stages
    assert probe.mp_probe_step_streams_bulk(*args, n, 4, 7, 0, err.data_ptr(), s) != 0  # does not fit
    assert probe.mp_probe_step_streams_bulk(params[1:].data_ptr(), *args[1:], n - TILE, 1, 4, 0, err.data_ptr(),
                                            s) != 0  # unaligned
    tile = probe.mp_probe_step_streams_bulk_tile
    assert tile(*args, n, 0, 1, 2, 0, err.data_ptr(), s) != 0  # no tile
    assert tile(*args, n, 96, 1, 2, 0, err.data_ptr(), s) != 0  # not a multiple of 64
    assert tile(*args, n, 3 * TILE, 1, 2, 0, err.data_ptr(), s) != 0  # n not whole tiles
    assert tile(*args, n, 4 * TILE, 1, 3, 0, err.data_ptr(), s) != 0  # 3 stages of 112 KB do not fit
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_bounded_mbarrier_wait_gives_up_and_reports(probe):
    """The staged kernels' mbarrier waits give up after one second of the
    global timer instead of spinning forever. Here every stage's barrier is
    told to expect 16 bytes more than its bulk load brings, so no phase ever
    completes (every byte lands; nothing faults): the kernel must end on its
    own within a few seconds, report the give-up in its error word, and leave
    the GPU usable (a normal probe afterwards moves its bytes exactly)."""
    tiles = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(2 * tiles * TILE * 14, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    rc = probe.mp_probe_bulk_timeout(buf.data_ptr(), tiles, err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, rc
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert int(err.item()) == 1
    assert 0.9 < elapsed < 30, elapsed  # one-second waits, not an endless spin
    test_bulk_copy_probe_copies_its_tiles(probe, 1, 7, 1)
