"""lcx_attention_noalloc, the attention entry point for callers that cannot allocate device
memory (for example a plugin whose host application owns all device allocations), against
lcx_attention with a caller workspace, through the C ABI.

Two calls in a row on different inputs, both of which use the fixed scratch array: the second
call checks that the array's leftover contents from the first do not leak into its result.
This file is collected last so that a run stopping at the first failure has run every other
test before it; it also passes alone in a fresh process."""
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
TOL = 1e-5   # the relative L2 tolerance of the attention parity tests


def case(seed, H, KV, hd, lengths, queries):
    rng = np.random.default_rng(seed)
    pages_per = [(n + PAGE - 1) // PAGE for n in lengths]
    n_pages = sum(pages_per) + 2
    pt = np.zeros((len(lengths), max(pages_per)), dtype=np.int32)
    perm, k = rng.permutation(n_pages), 0
    for s, n in enumerate(pages_per):
        pt[s, :n] = perm[k:k + n]
        k += n
    cells = n_pages * KV * PAGE * hd
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    host = dict(pt=pt, seq=np.array([s for s, _ in queries], np.int32), pos=np.array([p for _, p in queries], np.int32))
    return dict(
        host=host,
        q=dev(synth.normal(seed, 3, len(queries) * H * hd, 0.0, 0.2).reshape(len(queries), H * hd)),
        kc=dev(synth.normal(seed, 1, cells, 0.0, 1.0).astype(np.float16).reshape(n_pages, KV, PAGE, hd)),
        vc=dev(synth.normal(seed, 2, cells, 0.0, 1.0).astype(np.float16).reshape(n_pages, KV, PAGE, hd)),
        pt=dev(pt), seq=dev(np.array([s for s, _ in queries], np.int32)),
        pos=dev(np.array([p for _, p in queries], np.int32)), max_pos=max(p for _, p in queries), H=H, KV=KV, hd=hd)


def with_workspace(c):
    T = c["q"].shape[0]
    out = torch.full_like(c["q"], float("nan"))
    need = lcx.attention_workspace_size(T, c["H"], c["KV"], c["hd"], c["max_pos"])
    assert need > 0, "the case must exercise the scratch"
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert lcx.attention(c["q"], c["kc"], c["vc"], c["pt"], c["pos"], c["seq"], c["max_pos"], out, ws) == 0
    return out


def without_allocation(c):
    out = torch.full_like(c["q"], float("nan"))
    assert lcx.attention_noalloc(c["q"], c["kc"], c["vc"], c["pt"], c["pos"], c["seq"], c["max_pos"], out) == 0
    return out


def oracle_rows(c, rows):
    """The oracle's attention of query rows `rows`: the cells 0..pos of the query's sequence."""
    q, kc, vc = (c[k].cpu().numpy() for k in ("q", "kc", "vc"))
    h = c["host"]
    out = {}
    for t in rows:
        s, p = int(h["seq"][t]), int(h["pos"][t])
        idx = np.arange(p + 1)
        pages = h["pt"][s][idx // PAGE]
        K = kc[pages, :, idx % PAGE, :].astype(np.float64).reshape(p + 1, -1)
        Vv = vc[pages, :, idx % PAGE, :].astype(np.float64).reshape(p + 1, -1)
        out[t] = oracle.attend_gqa(q[t].astype(np.float64), K, Vv, c["H"], c["KV"], c["hd"])
    return out


def test_noalloc_matches_workspace_entry_on_two_calls():
    lcx.build()
    cases = [case(41, 32, 8, 128, [32896], [(0, 32895), (0, 20000)]),
             case(42, 4, 2, 64, [3000, 700, 64], [(0, 2999), (1, 699), (2, 63)])]
    for c in cases:
        got = without_allocation(c)
        ref = with_workspace(c)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        # the same kernel with the same split of the cells: bit for bit the same result
        assert torch.equal(got, ref)
        want = oracle_rows(c, range(got.shape[0]))
        g = got.double().cpu().numpy()
        for t, w in want.items():
            err = np.linalg.norm(g[t] - w) / np.linalg.norm(w)
            assert err <= TOL, (t, err)


def test_noalloc_scratch_covers_every_call_on_this_gpu():
    """The fixed array bounds what lcx_attention_noalloc can serve; a call needing more is
    refused on the host with LCX_INVALID. The split of the cell range keeps the scratch need at
    most about 2 x SMs x 8 query heads x (head_dim + 2) floats, so on this GPU every shape the
    entry point accepts fits: checked over the shapes (a bounded sweep), so that no caller of
    this GPU ever meets the refusal."""
    lcx.build()
    worst = 0
    for hd in (64, 128):
        for H, KV in ((32, 8), (8, 8), (64, 8), (32, 4), (4, 4), (8, 1), (16, 2), (64, 64)):
            for T in (1, 2, 3, 5, 8, 9, 16, 19, 33, 64, 152, 1024):
                for max_pos in (0, 63, 64, 1000, 4096, 32767, 262143):
                    worst = max(worst, lcx.attention_workspace_size(T, H, KV, hd, max_pos))
    assert 0 < worst <= lcx.LCX_ATTENTION_NOALLOC_SCRATCH_BYTES, worst
