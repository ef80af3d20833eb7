"""Parity of the attention step (lcx_attention, the kernel lcx_decode runs) with the oracle's
attention at the full sizes of the workloads: 32k-position long-context decode and 64-sequence
batched decode on the 8B shape, plus the tiny shape. K/V are random f16 cells scattered over
pages in a random order."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_ubatch_forward_gb300 as lcx  # noqa: E402

PAGE = 64


def make_case(seed, H, KV, hd, lengths, queries):
    """lengths: cells per sequence; queries: (seq, pos) pairs. Returns host and device arrays."""
    rng = np.random.default_rng(seed)
    n_seq = len(lengths)
    pages_per = [(n + PAGE - 1) // PAGE for n in lengths]
    n_pages = sum(pages_per) + 3
    max_pages = max(pages_per)
    perm = rng.permutation(n_pages)
    pt = np.zeros((n_seq, max_pages), dtype=np.int32)
    k = 0
    for s in range(n_seq):
        pt[s, :pages_per[s]] = perm[k:k + pages_per[s]]
        k += pages_per[s]
    kc = synth.normal(seed, 1, n_pages * KV * PAGE * hd, 0.0, 1.0).astype(np.float16).reshape(n_pages, KV, PAGE, hd)
    vc = synth.normal(seed, 2, n_pages * KV * PAGE * hd, 0.0, 1.0).astype(np.float16).reshape(n_pages, KV, PAGE, hd)
    T = len(queries)
    q = synth.normal(seed, 3, T * H * hd, 0.0, 0.2).reshape(T, H * hd)
    seq = np.array([s for s, _ in queries], dtype=np.int32)
    pos = np.array([p for _, p in queries], dtype=np.int32)
    return dict(pt=pt, kc=kc, vc=vc, q=q, seq=seq, pos=pos, H=H, KV=KV, hd=hd)


def oracle_out(c, t):
    s, p = int(c["seq"][t]), int(c["pos"][t])
    idx = np.arange(p + 1)
    pages = c["pt"][s][idx // PAGE]
    K = c["kc"][pages, :, idx % PAGE, :].astype(np.float64).reshape(p + 1, -1)
    V = c["vc"][pages, :, idx % PAGE, :].astype(np.float64).reshape(p + 1, -1)
    return oracle.attend_gqa(c["q"][t], K, V, c["H"], c["KV"], c["hd"])


def gpu_out(c, workspace="auto"):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    T = c["q"].shape[0]
    out = torch.full((T, c["H"] * c["hd"]), float("nan"), dtype=torch.float32, device="cuda")
    max_pos = int(c["pos"].max())
    need = lcx.attention_workspace_size(T, c["H"], c["KV"], c["hd"], max_pos)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda") if workspace == "auto" else workspace
    rc = lcx.attention(dev(c["q"]), dev(c["kc"]), dev(c["vc"]), dev(c["pt"]), dev(c["pos"]), dev(c["seq"]),
                       max_pos, out, ws)
    torch.cuda.synchronize()
    return rc, out.cpu().numpy().astype(np.float64)


def check(c, got, tol=1e-5):
    for t in range(got.shape[0]):
        ref = oracle_out(c, t)
        err = np.linalg.norm(got[t] - ref) / np.linalg.norm(ref)
        assert err <= tol, (t, err)


@pytest.fixture(scope="module", autouse=True)
def setup():
    lcx.build()
    oracle.set_threads()


def test_long_context_32k():
    c = make_case(31, 32, 8, 128, [32896], [(0, 32767), (0, 32895), (0, 0), (0, 4097)])
    rc, got = gpu_out(c)
    assert rc == 0
    check(c, got)


def test_multi_sequence_64():
    lengths = synth.multiseq_prompt_lengths(synth.CONFIGS["multiseq"], 64) + 1
    qs = [(s, int(n) - 1) for s, n in enumerate(lengths)]
    c = make_case(32, 32, 8, 128, lengths.tolist(), qs)
    rc, got = gpu_out(c)
    assert rc == 0
    check(c, got)


def test_tiny_shape_and_prefill_block():
    # 40 consecutive positions of one sequence (a prefill ubatch) plus a second sequence
    qs = [(0, p) for p in range(60, 100)] + [(1, 5)]
    c = make_case(33, 4, 2, 64, [100, 6], qs)
    rc, got = gpu_out(c)
    assert rc == 0
    check(c, got)


def test_small_workspace_is_rejected():
    c = make_case(34, 32, 8, 128, [4096], [(0, 4095)])
    need = lcx.attention_workspace_size(1, 32, 8, 128, 4095)
    assert need > 0
    rc, _ = gpu_out(c, workspace=torch.empty(need // 2, dtype=torch.uint8, device="cuda"))
    assert rc == lcx.LCX_INVALID
