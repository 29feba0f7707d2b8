"""Shard-on-read from a safetensors file onto the GPU, against the oracle's reader and shard.

"Tensor parallelism" page, §Load a sharded model: each rank reads only its
slice of each weight, straight to its device; §Loading performance: peak CPU
memory per rank stays far below the checkpoint's size.  Every loaded shard
must equal, byte for byte, the oracle's shard of the tensor the oracle reads
from the same file.
"""
import os
import resource

import numpy as np
import pytest
import torch

import tp_inputs
from oracle import st_oracle
from oracle import tp_oracle as O

pytestmark = pytest.mark.gpu

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")

DEV = "cuda"


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    tp.tp_device_status()


def host_bytes(t):
    torch.cuda.synchronize()
    return t.cpu().contiguous().view(torch.uint8).numpy().tobytes()


def matrix(arr, style):
    """The matrix view the loader shards: 1-D as [n, 1], N-D as [d0, d1*d2*...]."""
    if arr.ndim == 1:
        return arr.reshape(-1, 1)
    return arr.reshape(arr.shape[0], -1)


def want_shard(arr, style, p, r, splits=None):
    return np.ascontiguousarray(O.shard(matrix(arr, style), style, p, r, splits)).tobytes()


H, F, HEADS = 96, 288, 6       # [1,1,1,3,3] single-stream packing at mlp_ratio 3


def model_tensors(seed=0):
    rng = np.random.default_rng(seed)
    return [
        ("single.0.attn.to_qkv_mlp_proj.weight", "BF16", tp_inputs.random_bits(seed, 0, (3 * H + 2 * F, H))),
        ("single.0.attn.to_qkv_mlp_proj.bias", "BF16", tp_inputs.random_bits(seed, 1, (3 * H + 2 * F,))),
        ("single.0.attn.to_out.weight", "BF16", tp_inputs.random_bits(seed, 2, (H, H + F))),
        ("single.0.norm.weight", "F32", rng.standard_normal(H).astype(np.float32)),
        ("adaln.linear.weight", "F32", rng.standard_normal((6 * H, 4 * H)).astype(np.float32)),
        ("quant.codes", "I8", rng.integers(-128, 128, (48, 30), dtype=np.int8)),
        ("conv.weight", "F16", rng.standard_normal((12, 4, 3, 3)).astype(np.float16)),
    ]


# (name, style, splits, num_heads) -- the plan each tensor is loaded with.
PLAN = [
    ("single.0.attn.to_qkv_mlp_proj.weight", "colwise", [H, H, H, F, F], HEADS),
    ("single.0.attn.to_qkv_mlp_proj.bias", "colwise", [H, H, H, F, F], HEADS),
    ("single.0.attn.to_out.weight", "rowwise", [H, F], HEADS),
    ("adaln.linear.weight", "rowwise", None, 0),
    ("quant.codes", "colwise", None, 0),
    ("conv.weight", "colwise", None, 0),
]


READ_MODES = ["staged", "mapped"]


def open_file(path, staging, mode):
    """The file opened in `mode`; skips where mapped reads are not available on this device."""
    f = tp.SafetensorsFile(path, staging, read_mode=mode)
    try:
        got = f.read_mode_on_device()
    except tp.TPError as e:
        f.close()
        if mode == "mapped" and e.name == "TP_ERR_UNSUPPORTED":
            pytest.skip(f"mapped reads not available: {e}")
        raise
    assert got == mode
    return f


def test_auto_mode_takes_mapped_reads_where_available(tmp_path):
    path = str(tmp_path / "model.safetensors")
    tp_inputs.write_safetensors(path, model_tensors())
    with tp.SafetensorsFile(path, read_mode="mapped") as f:
        try:
            available = f.read_mode_on_device() == "mapped"
        except tp.TPError as e:
            assert e.name == "TP_ERR_UNSUPPORTED", e
            assert "mapped reads are not available" in str(e)
            available = False
    with tp.SafetensorsFile(path) as f:
        assert f.read_mode_on_device() == ("mapped" if available else "staged")


@pytest.mark.parametrize("mode", READ_MODES)
@pytest.mark.parametrize("staging", [0, 8192])
@pytest.mark.parametrize("p", [1, 2, 3, 6])
def test_every_rank_bit_exact(tmp_path, p, staging, mode):
    # staging 8192 bytes: every tensor crosses several staging buffers (chunk boundaries
    # inside rows for colwise, several row chunks for rowwise).
    path = str(tmp_path / "model.safetensors")
    tp_inputs.write_safetensors(path, model_tensors())
    ref, _ = st_oracle.read_safetensors(path)
    with open_file(path, staging, mode) as f:
        for name, style, splits, heads in PLAN:
            shards = f.shard_ranks(name, style, p, fused_splits=splits, num_heads=heads, device=DEV)
            for r, t in enumerate(shards):
                assert host_bytes(t) == want_shard(ref[name], style, p, r, splits), (name, p, r)
        # A replicated tensor: tp_degree 1.
        (full,) = f.shard_ranks("single.0.norm.weight", "colwise", 1, device=DEV)
        assert host_bytes(full) == ref["single.0.norm.weight"].tobytes()


@pytest.mark.parametrize("mode", READ_MODES)
def test_rank_subsets_and_given_outputs(tmp_path, mode):
    path = str(tmp_path / "model.safetensors")
    tp_inputs.write_safetensors(path, model_tensors(1))
    ref, _ = st_oracle.read_safetensors(path)
    p = 6
    with open_file(path, 16384, mode) as f:
        for name, style, splits, heads in PLAN[:4]:
            outs = f.shard_ranks(name, style, p, rank_begin=2, rank_count=3, fused_splits=splits, num_heads=heads,
                                 device=DEV)
            for i, t in enumerate(outs):
                assert host_bytes(t) == want_shard(ref[name], style, p, 2 + i, splits), (name, i)
        # Into caller-given buffers, on a side stream.
        name, style, splits, heads = PLAN[0]
        s = torch.cuda.Stream()
        bufs = [torch.full((3 * H // p + 2 * F // p, H), -1, dtype=torch.int16, device=DEV) for _ in range(p)]
        f.shard_ranks(name, style, p, fused_splits=splits, num_heads=heads, outs=bufs, stream=s)
        s.synchronize()
        for r, t in enumerate(bufs):
            assert host_bytes(t) == want_shard(ref[name], style, p, r, splits)


@pytest.mark.parametrize("mode", READ_MODES)
def test_shards_match_the_in_memory_extraction(tmp_path, mode):
    # Loading from the file and extracting from a device copy of the same weight give the
    # same shards: the two loading routes the page describes agree.
    w_in, w_out, _ = tp_inputs.single_stream_inputs(7, tokens=8, hidden=768, mlp_ratio=3)
    Hh, Ff = 768, 2304
    path = str(tmp_path / "block.safetensors")
    tp_inputs.write_safetensors(path, [("w_in", "BF16", w_in), ("w_out", "BF16", w_out)])
    p = 3
    with open_file(path, 0, mode) as f:
        a = f.shard_ranks("w_in", "colwise", p, fused_splits=[Hh, Hh, Hh, Ff, Ff], num_heads=6, device=DEV)
        b = f.shard_ranks("w_out", "rowwise", p, fused_splits=[Hh, Ff], num_heads=6, device=DEV)
    a2 = tp.tp_plan_shard_ranks(tp.bf16_from_bits(w_in, DEV), "colwise", p, 0, p, [Hh, Hh, Hh, Ff, Ff], 6, 0)
    b2 = tp.tp_plan_shard_ranks(tp.bf16_from_bits(w_out, DEV), "rowwise", p, 0, p, [Hh, Ff], 6, 0)
    for x, y in zip(a + b, a2 + b2):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def _hwm_reset_supported():
    try:
        with open("/proc/self/clear_refs", "w") as fh:
            fh.write("5")
        return True
    except OSError:
        return False


def _rss_anon_bytes():
    with open("/proc/self/status") as fh:
        for line in fh:
            if line.startswith("RssAnon:"):
                return int(line.split()[1]) * 1024
    return None


def _vm_hwm_bytes():
    with open("/proc/self/status") as fh:
        for line in fh:
            if line.startswith("VmHWM:"):
                return int(line.split()[1]) * 1024
    return resource.getrusage(resource.RUSAGE_SELF).ru_maxrss * 1024


@pytest.mark.slow
@pytest.mark.parametrize("mode", READ_MODES)
def test_large_weight_host_memory_stays_at_staging_size(tmp_path, mode):
    # A 302 MB packed to_out weight (hidden 6144, mlp_hidden 18432) loaded for all 4 ranks
    # with 8 MiB staging buffers.  Staged: the process's peak resident memory grows by about
    # the staging size, not by the weight's size.  Mapped: its anonymous memory does not grow
    # (the pages it reads are the page cache's, mapped in, not copies of them).
    Hh, Ff, p = 6144, 18432, 4
    path = str(tmp_path / "big.safetensors")
    w = tp_inputs.random_bits(9, 0, (Hh, Hh + Ff))
    w_in = tp_inputs.random_bits(9, 1, (3 * Hh + 2 * Ff, 1024))
    tp_inputs.write_safetensors(path, [("to_out", "BF16", w), ("in_proj", "BF16", w_in)])
    del w, w_in
    staging = 8 << 20
    outs_row = [torch.empty((Hh, (Hh + Ff) // p), dtype=torch.bfloat16, device=DEV) for _ in range(p)]
    outs_col = [torch.empty(((3 * Hh + 2 * Ff) // p, 1024), dtype=torch.bfloat16, device=DEV) for _ in range(p)]
    with open_file(path, staging, mode) as f:
        f.shard_ranks("to_out", "rowwise", p, fused_splits=[Hh, Ff], outs=outs_row)   # warm-up: staging allocated
        torch.cuda.synchronize()
        f.shard_ranks("in_proj", "colwise", p, fused_splits=[Hh, Hh, Hh, Ff, Ff], outs=outs_col)
        torch.cuda.synchronize()
        if mode == "staged" and not _hwm_reset_supported():
            pytest.skip("cannot reset the peak-RSS counter on this kernel")
        if mode == "mapped" and _rss_anon_bytes() is None:
            pytest.skip("no RssAnon line in /proc/self/status")
        base = _vm_hwm_bytes() if mode == "staged" else _rss_anon_bytes()
        f.shard_ranks("to_out", "rowwise", p, fused_splits=[Hh, Ff], outs=outs_row)
        f.shard_ranks("in_proj", "colwise", p, fused_splits=[Hh, Hh, Hh, Ff, Ff], outs=outs_col)
        torch.cuda.synchronize()
        grew = (_vm_hwm_bytes() if mode == "staged" else _rss_anon_bytes()) - base
    weight_bytes = Hh * (Hh + Ff) * 2
    assert grew < 4 * staging, (grew, weight_bytes)
    ref, _ = st_oracle.read_safetensors(path)
    rng = np.random.default_rng(3)
    for r in range(p):
        rows = np.sort(rng.choice(Hh, 64, replace=False))
        got = outs_row[r][torch.from_numpy(rows).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
        want = O.shard(ref["to_out"], "rowwise", p, r, [Hh, Ff])[rows]
        assert np.array_equal(got, want), r
        rows = np.sort(rng.choice((3 * Hh + 2 * Ff) // p, 64, replace=False))
        got = outs_col[r][torch.from_numpy(rows).to(DEV)].view(torch.int16).cpu().numpy().view(np.uint16)
        want = O.shard(ref["in_proj"], "colwise", p, r, [Hh, Hh, Hh, Ff, Ff])[rows]
        assert np.array_equal(got, want), r


@pytest.mark.parametrize("mode", READ_MODES)
def test_file_truncated_after_open_is_an_io_error(tmp_path, mode):
    # The header was checked at open; the data then shrinks under the handle.  Staged reads
    # come up short; mapped reads find the missing pages when they populate a range, on the
    # host, before the copy of that range is issued.
    path = str(tmp_path / "model.safetensors")
    w = tp_inputs.random_bits(4, 0, (1024, 512))
    tp_inputs.write_safetensors(path, [("w", "BF16", w)])
    f = open_file(path, 1 << 20, mode)
    try:
        size = os.path.getsize(path)
        os.truncate(path, size - 600 * 512 * 2)       # the last 600 rows are gone
        with pytest.raises(tp.TPError) as e:
            f.shard_ranks("w", "colwise", 2, device=DEV)
        assert e.value.name == "TP_ERR_IO", e.value
        torch.cuda.synchronize()
    finally:
        f.close()
