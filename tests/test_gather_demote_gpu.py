"""GPU parity of ekv_gather_prefill and ekv_demote_pages: bit-exact against the oracle."""

import numpy as np
import pytest

from mixed_precision_paged_gb300 import workloads as wl
from oracle import demote as odm
from oracle import gather as og

from _helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def run_gather(ekv_lib, torch, case, page_range, ws_pages, apply_scale=1):
    d = to_device(case)
    H, D = case.num_kv_heads, case.head_dim
    ws_k = torch.full((ws_pages, 16, H, D), float("nan"), dtype=torch.float16, device="cuda")
    ws_v = torch.full((ws_pages, 16, H, D), float("nan"), dtype=torch.float16, device="cuda")
    idx = torch.full((ws_pages,), -1, dtype=torch.int32, device="cuda")
    ctx = ekv_lib.Context(case.num_q_heads, H, D, 1)
    ekv_lib.ekv_gather_prefill(ctx.handle, d.k_pages, d.v_pages, case.v_page_stride, case.num_pages,
                               d.v_scales, case.scale_mode, d.page_mode, case.uniform_mode,
                               d.block_table, case.block_table.shape[1], case.batch, page_range,
                               ws_k, ws_v, idx, ws_pages, apply_scale)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    return ws_k.cpu().numpy(), ws_v.cpu().numpy(), idx.cpu().numpy()


@pytest.mark.parametrize("fmt,scale_mode,apply", [("e4m3", 0, 1), ("e4m3", 1, 1), ("mixed", 1, 1),
                                                  ("fp16", 0, 1), ("e4m3", 1, 0), ("mixed", 0, 1)])
@pytest.mark.parametrize("hkv,d", [(8, 128), (2, 64), (4, 128)])
def test_gather_bit_exact(ekv_lib, torch_cuda, fmt, scale_mode, apply, hkv, d):
    lens = [300, 40, 1000, 17]
    case = wl.make_decode_case(lens, hkv * 2, hkv, d, v_format=fmt, scale_mode=scale_mode,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 4, seed=21, poison=False)
    page_range = np.array([[2, 3, 40], [0, 0, 19], [3, 1, 1], [1, 0, 0], [2, 50, 13]])
    total = int(page_range[:, 2].sum())
    ws_k, ws_v, idx = run_gather(ekv_lib, torch_cuda, case, page_range, total + 3, apply)
    rk, rv, ri = og.gather_prefill(case.k_pages, case.v_pages, case.v_scales, scale_mode,
                                   case.page_mode, case.uniform_mode, case.block_table, page_range,
                                   apply_scale=bool(apply))
    assert np.array_equal(ws_k[:total].view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(ws_v[:total].view(np.uint16), rv.view(np.uint16))
    assert np.array_equal(idx[:total], ri)
    assert np.all(idx[total:] == -1)        # slots past the gathered pages untouched


def test_gather_many_ranges_chunked(ekv_lib, torch_cuda):
    lens = [16 * 3] * 300
    case = wl.make_decode_case(lens, 8, 4, 64, v_format="mixed", scale_mode=1,
                               pool_pages=900, seed=22, poison=False)
    page_range = np.array([[s, s % 3, 1 + (s % 2)] for s in range(300)])
    page_range[:, 2] = np.minimum(page_range[:, 2], 3 - page_range[:, 1])
    total = int(page_range[:, 2].sum())
    ws_k, ws_v, idx = run_gather(ekv_lib, torch_cuda, case, page_range, total)
    rk, rv, ri = og.gather_prefill(case.k_pages, case.v_pages, case.v_scales, 1, case.page_mode,
                                   0, case.block_table, page_range)
    assert np.array_equal(ws_k.view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(ws_v.view(np.uint16), rv.view(np.uint16))
    assert np.array_equal(idx, ri)


def run_demote(ekv_lib, torch, vb, ids, mode, H, D):
    v = torch.from_numpy(vb.copy()).cuda()
    m = torch.from_numpy(mode.copy()).cuda()
    sc = torch.zeros((vb.shape[0], H), dtype=torch.float32, device="cuda")
    pid = torch.from_numpy(np.asarray(ids, dtype=np.int32)).cuda()
    ctx = ekv_lib.Context(H, H, D, 1)
    ekv_lib.ekv_demote_pages(ctx.handle, v, vb.shape[1], vb.shape[0], pid, len(ids), m, sc)
    torch.cuda.synchronize()
    err = ctx.error()
    return v.cpu().numpy(), m.cpu().numpy(), sc.cpu().numpy(), err


@pytest.mark.parametrize("hkv,d,std", [(8, 128, 2 ** 0.5), (2, 64, 1.0), (4, 128, 1e-3), (1, 64, 300.0)])
def test_demote_bit_exact(ekv_lib, torch_cuda, hkv, d, std):
    rng = np.random.default_rng(31)
    P = 40
    x = (rng.standard_normal((P, 16, hkv, d)) * std).astype(np.float16)
    x[3] = 0
    x[5, :, 0] = -x[5, :, 0]
    vb = x.reshape(P, -1).view(np.uint8).copy()
    mode = np.zeros(P, dtype=np.uint8)
    mode[7] = 1                                   # already compact: skipped
    ids = rng.permutation(P)[:20].tolist() + [7, 3]
    v, m, sc, err = run_demote(ekv_lib, torch_cuda, vb, ids, mode, hkv, d)
    rv, rm, rs = odm.demote_pages(vb, ids, mode, np.zeros((P, hkv), np.float32), hkv, d)
    assert err == (0, 0)
    assert np.array_equal(m, rm)
    assert np.array_equal(v, rv)
    demoted = [p for p in set(ids) if mode[p] == 0]
    assert np.array_equal(sc[demoted], rs[demoted])


@pytest.mark.parametrize("P,n,hkv,d", [(4096, 4000, 8, 128), (160000, 158000, 1, 64)])
def test_demote_streams_many_pages_per_cta(ekv_lib, torch_cuda, P, n, hkv, d):
    """Enough pages that every CTA of the persistent demotion kernel cycles its slot
    ring many times (first case: ~13 pages per CTA through 3 slots), and (second case:
    more than 256 pages per CTA) restages its page-id table. Some pages are already
    compact and are skipped."""
    rng = np.random.default_rng(37)
    x = (rng.standard_normal((P, 16, hkv, d)) * 2 ** 0.5).astype(np.float16)
    vb = x.reshape(P, -1).view(np.uint8).copy()
    mode = np.zeros(P, dtype=np.uint8)
    mode[rng.choice(P, size=P // 50, replace=False)] = 1
    ids = rng.permutation(P)[:n]
    v, m, sc, err = run_demote(ekv_lib, torch_cuda, vb, ids, mode, hkv, d)
    rv, rm, rs = odm.demote_pages(vb, ids, mode, np.zeros((P, hkv), np.float32), hkv, d)
    assert err == (0, 0)
    assert np.array_equal(m, rm)
    assert np.array_equal(v, rv)
    demoted = np.array([p for p in ids if mode[p] == 0])
    assert np.array_equal(sc[demoted], rs[demoted])


def test_demote_then_gather_round_trip(ekv_lib, torch_cuda):
    import torch
    rng = np.random.default_rng(33)
    P, H, D = 24, 8, 128
    x = (rng.standard_normal((P, 16, H, D)) * 2 ** 0.5).astype(np.float16)
    vb = x.reshape(P, -1).view(np.uint8).copy()
    ids = rng.permutation(P)[:12]
    v, m, sc, err = run_demote(ekv_lib, torch_cuda, vb, ids, np.zeros(P, np.uint8), H, D)
    assert err == (0, 0)
    case = wl.DecodeCase(q=None, k_pages=rng.standard_normal((P, 16, H, D)).astype(np.float16),
                         v_pages=v, v_scales=sc, scale_mode=1, page_mode=m, uniform_mode=0,
                         block_table=np.arange(P, dtype=np.int32)[None, :],
                         seq_lens=np.array([16 * P], np.int32), num_q_heads=H, num_kv_heads=H,
                         head_dim=D)
    ws_k, ws_v, _ = run_gather(ekv_lib, torch, case, np.array([[0, 0, P]]), P)
    rv2, rm2, rs2 = odm.demote_pages(vb, ids, np.zeros(P, np.uint8), np.zeros((P, H), np.float32), H, D)
    _, ref_v, _ = og.gather_prefill(case.k_pages, rv2, rs2, 1, rm2, 0, case.block_table,
                                    np.array([[0, 0, P]]))
    assert np.array_equal(ws_v.view(np.uint16), ref_v.view(np.uint16))
    for p in range(P):
        if m[p] == 0:
            assert np.array_equal(ws_v[p].view(np.uint16), x[p].view(np.uint16))


def test_gather_chunks_back_to_back_under_pdl(ekv_lib, torch_cuda):
    """Gather calls back to back with the programmatic launch switched on (each next call
    reads its pages while the previous one drains): chunks into disjoint workspace
    regions and into the same region, a demotion and a cache-writer append in between
    (after which the gather runs in plain stream order); every call bit-exact against the
    oracle on the state it must see. More than 128 ranges per call also makes one call
    launch several kernels back to back."""
    torch = torch_cuda
    from oracle import writer as ow
    lens = [16 * 20 + 3] * 6 + [16 * 2] * 200
    case = wl.make_decode_case(lens, 16, 8, 128, v_format="mixed", scale_mode=1, seed=27, poison=False,
                               pool_pages=sum((l + 15) // 16 for l in lens) + 2, p_compact=0.4, p_base=0.2)
    d = to_device(case)
    H, D, B = 8, 128, case.batch
    ctx = ekv_lib.Context(16, H, D, B, pdl=True)
    chunks = [np.array([[b, 0, 21]]) for b in range(6)] + [np.array([[b, 0, 2] for b in range(6, 206)])]
    sizes = [int(c[:, 2].sum()) for c in chunks]
    W = sum(sizes)
    ws_k = torch.full((W, 16, H, D), float("nan"), dtype=torch.float16, device="cuda")
    ws_v = torch.full_like(ws_k, float("nan"))
    idx = torch.full((W,), -1, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    n_elem = 16 * H * D

    def gather(pr, off, n):
        ekv_lib.ekv_gather_prefill(ctx.handle, d.k_pages, d.v_pages, case.v_page_stride, case.num_pages,
                                   d.v_scales, 1, d.page_mode, 0, d.block_table, case.block_table.shape[1], B, pr,
                                   ws_k[off:off + n], ws_v[off:off + n], idx[off:off + n], n, 1, st)

    def check(k, v, pr, off, n, pool_v, pool_k, modes, scales):
        rk, rv, ri = og.gather_prefill(pool_k, pool_v, scales, 1, modes, 0, case.block_table, pr)
        assert np.array_equal(k[off:off + n].view(np.uint16), rk.view(np.uint16))
        assert np.array_equal(v[off:off + n].view(np.uint16), rv.view(np.uint16))

    for rep in range(20):                               # disjoint regions, no sync in between
        off = 0
        for pr, n in zip(chunks, sizes):
            gather(pr, off, n)
            off += n
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    k, v = ws_k.cpu().numpy(), ws_v.cpu().numpy()
    off = 0
    for pr, n in zip(chunks, sizes):
        check(k, v, pr, off, n, case.v_pages, case.k_pages, case.page_mode, case.v_scales)
        off += n
    assert np.array_equal(idx.cpu().numpy(), np.concatenate([np.arange(n) for n in sizes]))
    # the same region rewritten by consecutive calls: the last one wins
    for pr in chunks[:6]:
        gather(pr, 0, 21)
    torch.cuda.synchronize()
    check(ws_k.cpu().numpy(), ws_v.cpu().numpy(), chunks[5], 0, 21, case.v_pages, case.k_pages,
          case.page_mode, case.v_scales)
    # a demotion of sequence 0's TARGET pages, then at once a gather of them
    pages0 = case.block_table[0, :21]
    ids = np.array([p for p in pages0 if case.page_mode[p] == 0], np.int32)
    gather(chunks[1], 0, 21)
    ekv_lib.ekv_demote_pages(ctx.handle, d.v_pages, case.v_page_stride, case.num_pages,
                             torch.from_numpy(ids).cuda(), len(ids), d.page_mode, d.v_scales, st)
    gather(chunks[0], 0, 21)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    rv_pool, rm, rs = odm.demote_pages(case.v_pages, ids, case.page_mode, case.v_scales, H, D)
    check(ws_k.cpu().numpy(), ws_v.cpu().numpy(), chunks[0], 0, 21, rv_pool, case.k_pages, rm, rs)
    # a cache-writer append into sequence 1's last page, then at once a gather of it
    pos = np.full(B, -1, np.int32)
    pos[1] = lens[1] - 1                                # rewrite the last token of sequence 1
    kn = np.random.default_rng(28).standard_normal((B, H, D)).astype(np.float16)
    vn = np.random.default_rng(29).standard_normal((B, H, D)).astype(np.float16)
    gather(chunks[2], 0, 21)
    ekv_lib.ekv_append_kv(ctx.handle, torch.from_numpy(kn).cuda(), torch.from_numpy(vn).cuda(), d.k_pages,
                          d.v_pages, case.v_page_stride, case.num_pages, d.v_scales, 1, d.page_mode, 0,
                          d.block_table, case.block_table.shape[1], torch.from_numpy(pos).cuda(), B, st)
    gather(chunks[1], 0, 21)
    torch.cuda.synchronize()
    assert ctx.error() == (0, 0)
    k2, v2 = ow.append_token(case.k_pages, rv_pool, rs, 1, rm, 0, case.block_table, pos, kn, vn)
    check(ws_k.cpu().numpy(), ws_v.cpu().numpy(), chunks[1], 0, 21, v2, k2, rm, rs)
    assert n_elem == 16 * H * D
    ctx.close()
