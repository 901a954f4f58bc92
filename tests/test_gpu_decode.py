"""GPU parity of pass-Q decode (ring_attn_decode): a few query rows against a KV
cache kept in P stationary virtual shards; per-shard partials then the merge
kernel. Checked against the fp64 oracle evaluated at the query positions."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, host32
from online_softmax_merge_gb300.inputs import Workload, WORKLOADS, make_qkv
from oracle.attention import attention_at

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _check(q, k, v, P, q_pos0, layout, causal, scale=0.0):
    o, lse = ra.decode(q, k, v, P, q_pos0, layout, causal, scale)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    n_q, H = q.shape[1], q.shape[2]
    rows = np.arange(q_pos0, q_pos0 + n_q)
    O_ref, L_ref = attention_at(host32(q), rows, list(range(H)), H, host32(k), host32(v), causal,
                                scale=scale if scale > 0 else None)
    eo = float(np.abs(host32(o) - O_ref).max())
    el = float(np.abs(host32(lse) - L_ref).max())
    return eo, el


CASES = [
    # B, N, H, G, d, P, layout, causal, n_q, q_pos0 (None: the last n_q positions)
    (1, 4 * 700, 8, 2, 128, 4, "contiguous", True, 1, None),
    (2, 4 * 700, 8, 2, 128, 4, "striped", True, 3, None),
    (1, 3 * 1000, 4, 4, 128, 3, "contiguous", True, 2, 1234),     # mid-sequence: later shards empty
    (1, 8 * 512, 32, 8, 128, 8, "striped", True, 8, 2000),       # 32 rows per kv head
    (1, 2 * 300, 6, 2, 64, 2, "contiguous", False, 5, 0),
    (2, 5000, 2, 1, 64, 1, "contiguous", True, 4, None),         # P = 1, ragged chunks
    (1, 2 * 4500, 16, 1, 128, 2, "striped", True, 3, None),      # 48 rows: two row groups
    (1, 4 * 2600, 8, 2, 128, 2, "zigzag", True, 2, 5000),        # zigzag, chunks span halves
    (2, 8 * 512, 4, 1, 64, 4, "zigzag", True, 1, None),
    (1, 4 * 1100, 8, 2, 128, 4, "contiguous", True, 40, None),   # 160 rows: ten row groups
    (1, 2 * 9000, 4, 1, 128, 2, "contiguous", True, 1, None),    # 9000-key shards: two chunks
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_decode_matches_oracle(case):
    B, N, H, G, d, P, layout, causal, n_q, q_pos0 = case
    if q_pos0 is None:
        q_pos0 = N - n_q
    w = Workload("dec", B, N, H, G, d, P, layout, causal, seed=300 + CASES.index(case))
    _, k, v = make_qkv(w)
    g = torch.Generator().manual_seed(17)
    q = torch.randn((B, n_q, H, d), generator=g).to(torch.bfloat16)
    eo, el = _check(q.to(DEV), k.to(DEV), v.to(DEV), P, q_pos0, layout, causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


@pytest.mark.parametrize("scale", [0.04, 0.5])
def test_decode_with_explicit_scale(scale):
    w = Workload("decs", 1, 4 * 700, 8, 2, 128, 4, "striped", True, seed=340)
    _, k, v = make_qkv(w)
    g = torch.Generator().manual_seed(18)
    q = torch.randn((1, 2, 8, 128), generator=g).to(torch.bfloat16)
    eo, el = _check(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.seqlen - 2, w.layout, True, scale)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


def test_decode_one_token_on_the_128k_cache():
    w = WORKLOADS["c4"]
    _, k, v = make_qkv(w, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(18)
    q = torch.randn((w.batch, 1, w.heads, w.head_dim), generator=g, device=DEV).to(torch.bfloat16)
    eo, el = _check(q, k, v, w.P, w.seqlen - 1, w.layout, True)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


def test_decode_equals_fused_forward_rows():
    """The last rows of a full ring forward are the decode of those rows."""
    w = Workload("decfwd", 1, 4 * 384, 8, 2, 128, 4, "striped", True, seed=19)
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    of, lf = ra.fwd(q, k, v, w.P, w.layout, True)
    n_q = 5
    qd = q[:, -n_q:].contiguous()
    od, ld = ra.decode(qd, k, v, w.P, w.seqlen - n_q, w.layout, True)
    torch.cuda.synchronize()
    assert float((od.float() - of[:, -n_q:].float()).abs().max()) <= 2 * TOL_O
    assert float((ld - lf[:, :, -n_q:]).abs().max()) <= 2 * TOL_LSE


@pytest.mark.parametrize("case", [CASES[1], CASES[7]], ids=["striped", "zigzag"])
def test_decode_fp32_output(case):
    """Decode with O written as fp32 by the merge kernel: within the bar of the
    oracle, and its bf16 rounding is the bf16 call's output."""
    B, N, H, G, d, P, layout, causal, n_q, q_pos0 = case
    if q_pos0 is None:
        q_pos0 = N - n_q
    w = Workload("dec32", B, N, H, G, d, P, layout, causal, seed=350)
    _, k, v = (t.to(DEV) for t in make_qkv(w))
    g = torch.Generator().manual_seed(19)
    q = torch.randn((B, n_q, H, d), generator=g).to(torch.bfloat16).to(DEV)
    o32, l32 = ra.decode(q, k, v, P, q_pos0, layout, causal, out_dtype=torch.float32)
    o16, l16 = ra.decode(q, k, v, P, q_pos0, layout, causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    assert torch.equal(o16, o32.to(torch.bfloat16)) and torch.equal(l16, l32)
    rows = np.arange(q_pos0, q_pos0 + n_q)
    O_ref, L_ref = attention_at(host32(q), rows, list(range(H)), H, host32(k), host32(v), causal)
    assert float(np.abs(host32(o32) - O_ref).max()) <= TOL_O
    assert float(np.abs(host32(l32) - L_ref).max()) <= TOL_LSE
