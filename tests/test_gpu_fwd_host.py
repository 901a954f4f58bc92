"""ring_attn_fwd_host: the ring forward for inputs in host memory, pipelined one
(sequence, kv group) piece at a time through the workspace's device slots (inputs in
on the copy stream, outputs out on a stream of the call's own). Each piece is a
ring_attn_fwd call on its heads, so the results must equal the device path bit for
bit, whatever the number of slots."""
import pytest
import torch

from online_softmax_merge_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.mark.parametrize("B,H,G,layout,pinned", [
    (3, 4, 2, "contiguous", True), (1, 4, 2, "striped", True), (2, 4, 2, "zigzag", False),
    (4, 4, 2, "striped", False), (2, 3, 3, "contiguous", True), (2, 4, 1, "striped", True)])
def test_host_forward_equals_device_forward(B, H, G, layout, pinned):
    """Pieces of one kv group each (GQA, MHA: one head per piece, MQA: all heads)."""
    w = Workload("host", B, 4 * (2 * 128 + 40), H, G, 128, 4, layout, True, 400 + B + 10 * G)
    q, k, v = make_qkv(w)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h, l_h = ra.fwd_host(q, k, v, w.P, w.layout, w.causal, device=DEV)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    o_d, l_d = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("same_stream", [True, False])
def test_host_forward_after_prior_work_on_the_stream(same_stream):
    """The call's copies start only after work already enqueued on the stream (here:
    a device-to-host write into the host input the call then reads), whether the
    copies share the compute stream or run on the side stream."""
    w = Workload("host1", 2, 2 * 300, 2, 1, 64, 2, "contiguous", True, 410)
    q, k, v = (t.pin_memory() for t in make_qkv(w))
    q_dev = torch.randn(q.shape, device=DEV).to(torch.bfloat16)
    cur = torch.cuda.current_stream(DEV)
    torch.cuda._sleep(20_000_000)                 # keep the stream busy for a while
    q.copy_(q_dev, non_blocking=True)             # enqueued on the current stream
    o_h, l_h = ra.fwd_host(q, k, v, w.P, w.layout, w.causal, device=DEV,
                           copy_stream=cur if same_stream else None)
    torch.cuda.synchronize()
    o_d, l_d = ra.fwd(q_dev, k.to(DEV), v.to(DEV), w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


def test_host_forward_with_explicit_scale():
    w = Workload("hosts", 2, 4 * 200, 4, 2, 64, 4, "striped", True, 420)
    q, k, v = (t.pin_memory() for t in make_qkv(w))
    o_h, l_h = ra.fwd_host(q, k, v, w.P, w.layout, w.causal, scale=0.3, device=DEV)
    torch.cuda.synchronize()
    o_d, l_d = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal, 0.3)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("slots", [2, 3, 5])
def test_host_forward_with_fewer_slots_than_pieces(slots):
    """Eight pieces through 2, 3 or 5 slots: every slot is refilled while others are
    in use, at every stride."""
    w = Workload("hostslots", 4, 4 * 150, 4, 2, 128, 4, "contiguous", True, 430)
    q, k, v = (t.pin_memory() for t in make_qkv(w))
    full = ra.fwd_host_workspace_bytes(w.batch, w.seqlen, w.heads, w.kv_heads, w.head_dim,
                                       w.P, w.layout, w.causal)
    slot = full // 8                                      # 8 pieces: the default holds 8 slots
    ws = torch.empty(slots * slot, dtype=torch.uint8, device=DEV)
    o_h, l_h = ra.fwd_host(q, k, v, w.P, w.layout, w.causal, workspace=ws, device=DEV)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    o_d, l_d = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


@pytest.mark.parametrize("pinned", [(True, False, True, False, True), (False, True, False, True, False)])
def test_host_forward_with_mixed_page_locked_and_pageable_tensors(pinned):
    """Each host tensor goes its own way: page-locked ones through the SMs' copy
    kernels, pageable ones through the copy engines; the results are the same."""
    w = Workload("hostmix", 2, 4 * 200, 4, 2, 128, 4, "striped", True, 440)
    q, k, v = make_qkv(w)
    pq, pk, pv, po, pl = pinned
    q, k, v = (t.pin_memory() if p else t for t, p in ((q, pq), (k, pk), (v, pv)))
    o_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=po)
    l_h = torch.empty((w.batch, w.heads, w.seqlen), dtype=torch.float32, pin_memory=pl)
    ra.fwd_host(q, k, v, w.P, w.layout, w.causal, out=o_h, lse=l_h, device=DEV)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    o_d, l_d = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


def test_host_forward_on_views_inside_page_locked_buffers():
    """Tensors that start inside a larger page-locked allocation (not at its base)."""
    w = Workload("hostview", 1, 4 * 150, 4, 2, 64, 4, "contiguous", True, 450)
    q, k, v = make_qkv(w)
    big = torch.empty(q.numel() + 2 * k.numel() + 3 * 1024, dtype=torch.bfloat16).pin_memory()
    qv = big[1024:1024 + q.numel()].view(q.shape)
    kv_ = big[2048 + q.numel():2048 + q.numel() + k.numel()].view(k.shape)
    vv = big[3072 + q.numel() + k.numel():3072 + q.numel() + 2 * k.numel()].view(v.shape)
    qv.copy_(q)
    kv_.copy_(k)
    vv.copy_(v)
    o_h, l_h = ra.fwd_host(qv, kv_, vv, w.P, w.layout, w.causal, device=DEV)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    o_d, l_d = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())


def test_host_mapped_sees_page_locked_memory_and_views_inside_it():
    """The query behind the choice between copy kernels and copy engines."""
    pinned = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
    assert ra.host_mapped(pinned, DEV)
    assert ra.host_mapped(pinned[4096:8192], DEV)
    assert not ra.host_mapped(torch.empty(1 << 20, dtype=torch.uint8), DEV)
    with pytest.raises(ValueError):
        ra.host_mapped(pinned.to(DEV), DEV)
    lib = ra.load()
    assert lib.ring_attn_host_mapped(None, 16) == 0
    assert lib.ring_attn_host_mapped(pinned.data_ptr(), 0) == 0
    assert lib.ring_attn_host_mapped(pinned.data_ptr() + 1, 16) == 0      # not 4-byte aligned


def test_host_mapped_refuses_a_range_with_an_unmapped_hole():
    """Two registered 2 MiB ranges of one pageable buffer with 2 MiB between them:
    the first and last byte of the span are mapped, its middle is not, so the span
    must go through the copy engines. Only registers memory and queries attributes."""
    MB = 1 << 20
    buf = torch.empty(9 * MB, dtype=torch.uint8)
    off = (-buf.data_ptr()) % MB
    a0 = buf.data_ptr() + off
    cr = torch.cuda.cudart()
    flags = 3   # cudaHostRegisterPortable | cudaHostRegisterMapped
    torch.cuda.synchronize(DEV)
    r1 = int(cr.cudaHostRegister(a0, 2 * MB, flags))
    r2 = int(cr.cudaHostRegister(a0 + 4 * MB, 2 * MB, flags)) if r1 == 0 else -1
    try:
        if r1 != 0 or r2 != 0:
            pytest.skip(f"cudaHostRegister returned {r1}, {r2}")
        first, second = buf[off:off + 2 * MB], buf[off + 4 * MB:off + 6 * MB]
        if not (ra.host_mapped(first, DEV) and ra.host_mapped(second, DEV)):
            pytest.skip("registered memory is not mapped at its host address on this device")
        assert not ra.host_mapped(buf[off:off + 6 * MB], DEV)
        assert not ra.host_mapped(buf[off + MB:off + 5 * MB], DEV)
        assert not ra.host_mapped(buf[off:off + 2 * MB + 4096], DEV)     # runs past the end
    finally:
        if r1 == 0:
            cr.cudaHostUnregister(a0)
        if r2 == 0:
            cr.cudaHostUnregister(a0 + 4 * MB)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_forward_fp32_output_equals_device_forward(pinned):
    """O written as fp32 into host memory (pieces' strided output copies of 4-byte
    elements) equals the device forward's fp32 output bit for bit."""
    w = Workload("host32", 2, 4 * (128 + 40), 4, 2, 128, 4, "striped", True, 430)
    q, k, v = make_qkv(w)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h, l_h = ra.fwd_host(q, k, v, w.P, w.layout, w.causal, device=DEV,
                           out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    assert o_h.dtype == torch.float32 and o_h.device.type == "cpu"
    o_d, l_d = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal,
                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())
