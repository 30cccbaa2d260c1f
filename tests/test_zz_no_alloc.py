"""kvq_decode_attention_noalloc against kvq_decode_attention.

The no-allocation entry point serves callers that cannot allocate device
memory when they run attention (an engine that owns all GPU memory in its own
pool, or a path that must stay out of the allocator), so they keep the packed
cache in their own buffers.  This test builds such buffers from a cache's
export, in the page layout include/kvq.h documents, and checks two calls in a
row (different queries) against the regular entry point on the same cache,
within the attention tolerance the other GPU tests use.  The file name makes
pytest collect it last.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _r16(x):
    return (x + 15) // 16 * 16


def _unpack_rows(words, n, bits):
    """Token-major bitstream rows [T][n*bits/32] u32 -> codes [T][n]."""
    out = np.zeros((words.shape[0], n), np.uint32)
    for c in range(n):
        b = c * bits
        v = words[:, b // 32] >> np.uint32(b % 32)
        if b % 32 + bits > 32:
            v = v | (words[:, b // 32 + 1] << np.uint32(32 - b % 32))
        out[:, c] = v & np.uint32((1 << bits) - 1)
    return out


def _fragment_words(codes, bits, keys):
    """Codes of one page [R][128] in the fragment order include/kvq.h describes for 2- and
    4-bit codes: per 16-token tile and lane l = 4g + t, 2*bits words; pair j of a word holds
    its first code at bits [bits*j, ...) and its second at [16 + bits*j, ...)."""
    R = codes.shape[0]
    words = np.zeros((R // 16, 32, 2 * bits), np.uint32)
    for tile in range(R // 16):
        for lane in range(32):
            g, t = lane // 4, lane % 4
            for w in range(2 * bits):
                word = 0
                for j in range(16 // bits):
                    if keys:  # word w = r*bits + u: token 16*tile + g + 8r, channels c, c + 1
                        r, u = divmod(w, bits)
                        tok = 16 * tile + g + 8 * r
                        c = 16 * (u * (8 // bits) + j // 2) + 8 * (j % 2) + 2 * t
                        first, second = codes[tok, c], codes[tok, c + 1]
                    else:  # word w = r*(bits/2) + u: channel ch of tokens s, s + 1
                        r, u = divmod(w, bits // 2)
                        ch = 16 * (u * (16 // bits) + j) + g + 8 * (r % 2)
                        s = 16 * tile + 8 * (r // 2) + 2 * t
                        first, second = codes[s, ch], codes[s + 1, ch]
                    word |= int(first) << (bits * j) | int(second) << (16 + bits * j)
                words[tile, lane, w] = word
    return words.reshape(-1)


def _pages_and_window(cache, w, spare_pages=3):
    """Caller-owned copies of the cache: pages [units][Tq/R + spare_pages][page_bytes] (the unit stride
    is larger than the pages in use) and window [units][R][D]."""
    T, Tq, n_r = cache.state()
    R, D, G, nsp, bk, bv = w.residual, w.head_dim, w.group, w.k_sparse, w.k_bits, w.v_bits
    off_km = _r16(R * D * bk // 8)
    off_vc = off_km + _r16((R // G) * D * 4)
    off_vm = off_vc + _r16(R * D * bv // 8)
    off_si = off_vm + _r16(R * (D // G) * 4)
    off_sv = off_si + _r16(R * nsp)
    page_bytes = off_sv + _r16(R * nsp * 2)
    units = w.batch * w.kv_heads
    n_pages = Tq // R
    pages = np.zeros((units, n_pages + spare_pages, page_bytes), np.uint8)
    win_k = np.zeros((units, R, D), np.uint16)
    win_v = np.zeros((units, R, D), np.uint16)
    frag = bk in (2, 4) and bv in (2, 4) and not w.rope
    for u in range(units):
        b, kvh = divmod(u, w.kv_heads)
        st = cache.export_unit(b, kvh)
        for p in range(n_pages):
            pg = pages[u, p]
            kc = st["kcodes"][p * R:(p + 1) * R]
            vc = st["vcodes"][p * R:(p + 1) * R]
            if frag:
                kc = _fragment_words(_unpack_rows(kc, D, bk), bk, keys=True)
                vc = _fragment_words(_unpack_rows(vc, D, bv), bv, keys=False)
            pg[0:R * D * bk // 8] = kc.view(np.uint8).ravel()
            km = st["kz"][p * R // G:(p + 1) * R // G].astype(np.uint32) | (
                st["ks"][p * R // G:(p + 1) * R // G].astype(np.uint32) << 16)
            pg[off_km:off_km + km.nbytes] = km.view(np.uint8).ravel()
            pg[off_vc:off_vc + R * D * bv // 8] = vc.view(np.uint8).ravel()
            vm = st["vz"][p * R:(p + 1) * R].astype(np.uint32) | (st["vs"][p * R:(p + 1) * R].astype(np.uint32) << 16)
            pg[off_vm:off_vm + vm.nbytes] = vm.view(np.uint8).ravel()
            if nsp:
                pg[off_si:off_si + R * nsp] = st["sp_idx"][p * R:(p + 1) * R].ravel()
                pg[off_sv:off_sv + R * nsp * 2] = st["sp_val"][p * R:(p + 1) * R].view(np.uint8).ravel()
        win_k[u, :n_r] = st["wk"]
        win_v[u, :n_r] = st["wv"]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    return dev(pages), n_pages + spare_pages, dev(win_k), dev(win_v), T


@pytest.mark.parametrize("case", ["mha-2bit", "gqa-rope-sparse-3bit", "gqa4-2bit-shrunk-grid"])
def test_noalloc_matches_regular_decode_twice(case):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    if case == "mha-2bit":
        w = synth.WORKLOADS[1].scaled(batch=2, kv_heads=4, q_heads=4, prefill_tokens=700, decode_steps=2)
    elif case == "gqa-rope-sparse-3bit":
        w = synth.WORKLOADS[4].scaled(batch=1, kv_heads=2, q_heads=8, prefill_tokens=900, decode_steps=2)
    else:
        # 72 units of four query heads (the tensor-core kernel, 16 warps): on a 152-SM GPU the full
        # resident grid needs 16 * (ceil(152/72) + 2) = 80 slots per head, 12 MB of partials, more
        # than the 8 MiB array holds, so the call lowers the grid until they fit
        w = synth.WORKLOADS[3].scaled(batch=9, kv_heads=8, q_heads=32, prefill_tokens=300, decode_steps=2)
    K = synth.keys(w)
    V = synth.values(w)
    T0 = w.prefill_tokens
    cache = kvq.KVCache.for_workload(w)
    cache.prefill_quantize(torch.from_numpy(np.ascontiguousarray(K[:, :, :T0])).cuda(),
                           torch.from_numpy(np.ascontiguousarray(V[:, :, :T0])).cuda())
    cache.append(torch.from_numpy(np.ascontiguousarray(K[:, :, T0])).cuda(),
                 torch.from_numpy(np.ascontiguousarray(V[:, :, T0])).cuda())
    pages, n_pages, win_k, win_v, T = _pages_and_window(cache, w)
    for step in range(2):  # two calls in a row; the shared scratch keeps the previous call's contents
        q = torch.from_numpy(synth.queries(w, step)).cuda()
        ref = cache.decode_attention(q)
        out = torch.full_like(q, float("nan"))
        kvq.kvq.kvq_decode_attention_noalloc(cache.cfg, pages, n_pages, win_k, win_v, T, q, out)
        torch.cuda.synchronize()
        err = oracle.max_rel_err(out.float().cpu().numpy().reshape(-1, w.head_dim),
                                 ref.float().cpu().numpy().reshape(-1, w.head_dim).astype(np.float64))
        assert err <= TOL, (case, step, err)
        assert kvq.kvq.kvq_noalloc_sync_status() == 0  # no device-side wait ran out
    assert cache.sync_status() == 0
    cache.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    cfg = kvq.make_config(256, 32, 128, 128, 1024, 2, 2, 32, 128)  # 32768 query heads: partials exceed 8 MiB
    buf = torch.zeros(64, dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq.kvq_decode_attention_noalloc(cfg, buf, 8, buf, buf, 1000, buf, buf)
    assert e.value.status == kvq.kvq.KVQ_ERR_CAPACITY
