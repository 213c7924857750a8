"""gla_fwd_noalloc: the forward for callers that cannot allocate device memory.

Some hosts hand all device memory to their own pool and must account for every byte, and
some call from latency-critical code where a cudaMalloc / cudaFree (which synchronises the
whole device) is not allowed. For them the library offers gla_fwd_noalloc, which takes the
tensor-core path's scratch from a fixed array compiled into the library. These tests check,
through the C ABI, that its results match the fp64 oracle and gla_fwd (bf16 parity
tolerance) on two calls in a row that reuse the array, that its automatic split steps down
to the largest one whose scratch fits, and that a request whose scratch does not fit is
refused before anything runs. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from parity import assert_close

MAX_SCRATCH = 16 << 20          # GLA_NOALLOC_SCRATCH_BYTES
PER_SEGMENT_HEAD = (2 * 128 * 128 + 128) * 4


def _lib():
    from chunkwise_recurrent_prefill_gb300 import build_ext
    from chunkwise_recurrent_prefill_gb300.gla import load_library
    build_ext.build()
    return load_library()


def _raw_call(lib, B, T, H, seq_splits, addr=0x1000000000):
    """Host-side checks only: q is NULL, so even a call that got past the scratch checks would
    be refused (GLA_ERR_NULL_ARG) before anything launched; the other pointers are fake,
    far-apart addresses that nothing dereferences."""
    p = lambda i: ctypes.c_void_p(addr * (i + 1))  # noqa: E731
    return lib.gla_fwd_noalloc(None, p(1), p(2), p(3), ctypes.c_float(1.0), None, p(4), None,
                               B, T, H, 128, 128, seq_splits, None)


def test_noalloc_host_checks():
    lib = _lib()
    assert _raw_call(lib, 1, 1024, 16, -1) == 10                       # GLA_ERR_BAD_OPTION
    # 16 heads x 8 extra segments x 131584 B = 16.8 MB > 16 MiB: refused on the host
    assert 16 * 8 * PER_SEGMENT_HEAD > MAX_SCRATCH
    assert _raw_call(lib, 1, 1024, 16, 9) == 9                         # GLA_ERR_WORKSPACE
    detail = lib.gla_last_error_detail().decode()
    assert str(16 * 8 * PER_SEGMENT_HEAD) in detail and str(MAX_SCRATCH) in detail


def _inputs(B, T, H, seed, with_h0=True, D=128):
    from chunkwise_recurrent_prefill_gb300.workloads import make_inputs, small
    return make_inputs(small("noalloc", B=B, T=T, H=H, io="bf16", seed=seed, with_h0=with_h0,
                             Dk=D, Dv=D), torch.device("cuda:0"))


def _oracle(x):
    import oracle
    cpu = lambda t: None if t is None else t.cpu()  # noqa: E731
    return oracle.recurrent(cpu(x["q"]), cpu(x["k"]), cpu(x["v"]), cpu(x["g"]), x["scale"],
                            cpu(x["h0"]))


def _compare(x, seq_splits):
    """gla_fwd_noalloc against the fp64 oracle and against gla_fwd (same split request), both
    at the bf16 parity tolerance. Returns the noalloc outputs."""
    from chunkwise_recurrent_prefill_gb300 import gla_fwd, gla_fwd_noalloc, last_device_status
    B, T, H, D = x["q"].shape
    o = torch.empty((B, T, H, D), dtype=torch.bfloat16, device="cuda:0")
    hT = torch.empty((B, H, D, D), dtype=torch.float32, device="cuda:0")
    gla_fwd_noalloc(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], o=o, hT=hT,
                    seq_splits=seq_splits)
    torch.cuda.synchronize()
    assert last_device_status() == 0
    o_fwd, h_fwd = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"],
                           return_state=True, seq_splits=seq_splits)
    torch.cuda.synchronize()
    o_ref, h_ref = _oracle(x)
    o_np, h_np = o.float().cpu().numpy(), hT.cpu().numpy()
    assert_close(o_np, o_ref, "bf16", "o(noalloc) vs oracle")
    assert_close(h_np, h_ref, "bf16", "hT(noalloc) vs oracle")
    assert_close(o_np, o_fwd.float().cpu().numpy(), "bf16", "o(noalloc) vs gla_fwd")
    assert_close(h_np, h_fwd.cpu().numpy(), "bf16", "hT(noalloc) vs gla_fwd")
    return o, hT


@pytest.mark.gpu
def test_noalloc_matches_gla_fwd_two_calls():
    from chunkwise_recurrent_prefill_gb300.gla import launch_counter, workspace_size
    _lib()
    # first call: 4 heads split in 5 segments (2.1 MB of scratch)
    assert 0 < workspace_size(1, 2048, 4, path="tc", seq_splits=5) <= MAX_SCRATCH
    n0 = launch_counter()
    _compare(_inputs(1, 2048, 4, seed=41), seq_splits=5)
    assert launch_counter() - n0 == 3 + 3          # state + scan + output, for each entry
    # second call right after, another shape, automatic split; the array keeps the first
    # call's contents, which must not matter
    assert workspace_size(2, 1000, 3) > 0
    _compare(_inputs(2, 1000, 3, seed=42), seq_splits=0)


@pytest.mark.gpu
def test_noalloc_oversize_refused_and_auto_split_capped():
    from chunkwise_recurrent_prefill_gb300 import GLAError, gla_fwd_noalloc
    from chunkwise_recurrent_prefill_gb300.gla import workspace_size
    _lib()
    x = _inputs(1, 16384, 16, seed=43)
    o = torch.full((1, 16384, 16, 128), 7.0, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(GLAError) as e:
        gla_fwd_noalloc(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], o=o, seq_splits=9)
    assert e.value.status == 9 and "static scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((o.float() == 7.0).all())            # nothing ran
    # gla_fwd's automatic split wants more scratch than the array holds here; the
    # automatic split of gla_fwd_noalloc is capped to fit and still matches gla_fwd
    assert workspace_size(1, 16384, 16) > MAX_SCRATCH
    _compare(x, seq_splits=0)


@pytest.mark.gpu
def test_noalloc_auto_split_one_head_long_sequence():
    """One head of 16384 tokens: gla_fwd would cut it into 152 segments (19.9 MB of scratch).
    The automatic split of gla_fwd_noalloc steps down from there to the largest count that fits
    the 16 MiB array: 128 segments (127 x 131584 B). Its outputs are then bit for bit those of
    gla_fwd with seq_splits=128 (same kernels, same split, deterministic)."""
    from chunkwise_recurrent_prefill_gb300 import gla_fwd
    from chunkwise_recurrent_prefill_gb300.gla import workspace_size
    _lib()
    assert workspace_size(1, 16384, 1) > MAX_SCRATCH
    assert workspace_size(1, 16384, 1, seq_splits=128) <= MAX_SCRATCH
    assert workspace_size(1, 16384, 1, seq_splits=129) > MAX_SCRATCH
    x = _inputs(1, 16384, 1, seed=44)
    o, hT = _compare(x, seq_splits=0)
    o128, h128 = gla_fwd(x["q"], x["k"], x["v"], x["g"], x["scale"], x["h0"], return_state=True,
                         seq_splits=128)
    torch.cuda.synchronize()
    assert torch.equal(o, o128) and torch.equal(hT, h128)


@pytest.mark.gpu
def test_noalloc_head_pairs_d64():
    """Head dims 64 with an even head count run as head pairs of dims 128: the split and its
    scratch are those of the pair view. Here gla_fwd cuts each of the 8 pairs into 19 segments
    (18.9 MB of scratch), so the automatic split of gla_fwd_noalloc is capped to fit the
    array; the results still match the oracle and gla_fwd."""
    from chunkwise_recurrent_prefill_gb300.gla import workspace_size
    _lib()
    assert workspace_size(1, 4096, 16, Dk=64, Dv=64) == 8 * 18 * 131584 > MAX_SCRATCH
    _compare(_inputs(1, 4096, 16, seed=45, D=64), seq_splits=0)
