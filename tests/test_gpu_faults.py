"""Failure paths on the GPU, made to happen without a fault.

* Device-side time limits: every page and stage wait of the decode kernels gives up after a limit,
  records an error and lets the kernel finish.  kvq_test_inject leaves one page of every CTA's
  slice uncopied and shortens the limit to 1 ms, so the waits for that page run out: the call must
  come back quickly, kvq_sync_status must report KVQ_ERR_CUDA, and the context must stay usable (a
  new cache then decodes correctly).  Both decode kernels (tensor-core and CUDA-core).
* Out of memory in kvq_create: a caller allocator (kvq_set_device_allocator) that fails on its
  n-th call makes kvq_create return KVQ_ERR_OOM, and every block it had handed out is given back.
* The debug build (kernels check their buffer bounds, canaries follow every cache buffer): parity
  cases through it in a child process, then kvq_debug_check finds the error word clean and every
  canary intact.
"""
import ctypes
import os
import subprocess
import sys
import time

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = 2e-3


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _filled_cache(w):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    K, V = synth.keys(w), synth.values(w)
    T0 = w.prefill_tokens
    cache = kvq.KVCache.for_workload(w)
    cache.prefill_quantize(_dev(K[:, :, :T0]), _dev(V[:, :, :T0]))
    cache.append(_dev(K[:, :, T0]), _dev(V[:, :, T0]))
    return cache, K, V


def _check_against_oracle(w, out, K, V, q):
    T0 = w.prefill_tokens
    out = out.float().cpu().numpy().astype(np.float64)
    for b in range(w.batch):
        for kvh in range(w.kv_heads):
            u = oracle.OracleUnit.for_workload(w)
            u.prefill(K[b, kvh, :T0], V[b, kvh, :T0])
            u.append(K[b, kvh, T0], V[b, kvh, T0])
            hs = slice(kvh * w.group_q, (kvh + 1) * w.group_q)
            err = oracle.max_rel_err(out[b, hs], u.attention(q[b, hs], w.softmax_scale))
            assert err <= TOL, (b, kvh, err)


CASES = {
    # tensor-core kernel: 2-bit codes, keys stored after RoPE
    "mma": synth.WORKLOADS[1].scaled(batch=2, kv_heads=4, q_heads=4, prefill_tokens=1500, decode_steps=1),
    # CUDA-core kernel: 3-bit codes, keys rotated at decode, sparse entries
    "cuda-core": synth.WORKLOADS[4].scaled(batch=1, kv_heads=2, q_heads=8, prefill_tokens=1500, decode_steps=1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_wait_runs_out_and_is_reported(case):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = CASES[case]
    cache, K, V = _filled_cache(w)
    assert cache.sync_status() == 0
    q = _dev(synth.queries(w, 0))
    kvq.kvq.kvq_test_inject(cache.handle, 0, 1_000_000)  # page 0 of every slice never arrives; 1 ms limit
    t0 = time.perf_counter()
    cache.decode_attention(q)
    st = cache.sync_status()
    elapsed = time.perf_counter() - t0
    assert st == kvq.kvq.KVQ_ERR_CUDA
    assert elapsed < 1.0, elapsed  # the 1 ms limit ended the waits, not the 2 s default
    # the cache stays broken; the context does not: a new cache decodes correctly
    with pytest.raises(kvq.KVQError):
        cache.decode_attention(q)
    cache.close()
    torch.cuda.synchronize()
    fresh, K, V = _filled_cache(w)
    out = fresh.decode_attention(q)
    assert fresh.sync_status() == 0
    _check_against_oracle(w, out, K, V, synth.queries(w, 0))
    fresh.close()


def test_test_hook_arguments():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = CASES["mma"]
    cache = kvq.KVCache.for_workload(w)
    for bad in ((-2, 0), (0, -1)):
        with pytest.raises(kvq.KVQError) as e:
            kvq.kvq.kvq_test_inject(cache.handle, *bad)
        assert e.value.status == kvq.kvq.KVQ_ERR_INVALID_ARG
    kvq.kvq.kvq_test_inject(cache.handle, -1, 0)  # normal operation
    cache.close()


class _Pool:
    """A caller allocator over torch's caching allocator that fails on its n-th call."""

    def __init__(self, fail_at=None):
        import bit_asymmetric_kv_kvq_gb300 as kvq
        self.fail_at, self.calls, self.live = fail_at, 0, {}
        self.alloc_fn = kvq.kvq.KVQ_ALLOC_FN(self._alloc)
        self.free_fn = kvq.kvq.KVQ_FREE_FN(self._free)

    def _alloc(self, nbytes, device, user):
        self.calls += 1
        if self.fail_at is not None and self.calls == self.fail_at:
            return None
        ptr = torch.cuda.caching_allocator_alloc(nbytes, device)
        self.live[ptr] = nbytes
        return ptr

    def _free(self, ptr, device, user):
        assert ptr in self.live, "freed a block the pool did not hand out"
        del self.live[ptr]
        torch.cuda.caching_allocator_delete(ptr)


def test_create_out_of_memory_frees_what_it_allocated():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = CASES["mma"]
    n_blocks = None
    try:
        pool = _Pool()
        kvq.kvq.kvq_set_device_allocator(pool.alloc_fn, pool.free_fn)
        cache = kvq.KVCache.for_workload(w)
        n_blocks = pool.calls
        assert n_blocks >= 4 and len(pool.live) == n_blocks
        cache.close()
        assert pool.live == {}
        for n in range(1, n_blocks + 1):  # fail the first, second, ... allocation
            pool = _Pool(fail_at=n)
            kvq.kvq.kvq_set_device_allocator(pool.alloc_fn, pool.free_fn)
            with pytest.raises(kvq.KVQError) as e:
                kvq.KVCache.for_workload(w)
            assert e.value.status == kvq.kvq.KVQ_ERR_OOM
            assert pool.live == {}, n  # nothing left allocated
    finally:
        kvq.kvq.kvq_set_device_allocator(None, None)


def test_cache_on_a_caller_allocator_decodes_like_the_default():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = CASES["mma"]
    pool = _Pool()
    try:
        kvq.kvq.kvq_set_device_allocator(pool.alloc_fn, pool.free_fn)
        cache, K, V = _filled_cache(w)
    finally:
        kvq.kvq.kvq_set_device_allocator(None, None)
    q = synth.queries(w, 0)
    out = cache.decode_attention(_dev(q))
    assert cache.sync_status() == 0
    _check_against_oracle(w, out, K, V, q)
    cache.close()
    assert pool.live == {}
    with pytest.raises(kvq.KVQError) as e:  # one of the pair alone is refused
        kvq.kvq.kvq_set_device_allocator(pool.alloc_fn, None)
    assert e.value.status == kvq.kvq.KVQ_ERR_INVALID_ARG


_DEBUG_CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import bit_asymmetric_kv_kvq_gb300 as kvq
import oracle, synth
assert kvq.kvq.LIB_PATH.endswith("libkvq_debug.so")
cases = [synth.WORKLOADS[1].scaled(batch=2, kv_heads=4, q_heads=4, prefill_tokens=300, decode_steps=130),
         synth.WORKLOADS[3].scaled(batch=2, kv_heads=2, q_heads=8, prefill_tokens=400, decode_steps=3),
         synth.WORKLOADS[4].scaled(batch=1, kv_heads=2, q_heads=8, prefill_tokens=500, decode_steps=3),
         synth.WORKLOADS[2].scaled(batch=2, kv_heads=2, q_heads=2, prefill_tokens=260, decode_steps=2)]
dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
for w in cases:
    K, V = synth.keys(w), synth.values(w)
    T0 = w.prefill_tokens
    cache = kvq.KVCache.for_workload(w)
    cache.prefill_quantize(dev(K[:, :, :T0]), dev(V[:, :, :T0]))
    for i in range(w.decode_steps):  # fused steps across a flush
        q = synth.queries(w, i)
        out = cache.decode_step(dev(K[:, :, T0 + i]), dev(V[:, :, T0 + i]), dev(q)).float().cpu().numpy()
    T = T0 + w.decode_steps
    for b in range(w.batch):
        for kvh in range(w.kv_heads):
            u = oracle.OracleUnit.for_workload(w)
            u.prefill(K[b, kvh, :T0], V[b, kvh, :T0])
            for i in range(w.decode_steps):
                u.append(K[b, kvh, T0 + i], V[b, kvh, T0 + i])
            got, ref = cache.export_unit(b, kvh), u.stores()
            assert all(np.array_equal(got[k], ref[k]) for k in ref), (w.name, b, kvh)
            hs = slice(kvh * w.group_q, (kvh + 1) * w.group_q)
            err = oracle.max_rel_err(out[b, hs].astype(np.float64), u.attention(q[b, hs], w.softmax_scale))
            assert err <= 2e-3, (w.name, b, kvh, err)
    assert kvq.kvq.kvq_debug_check(cache.handle) == 0, w.name  # error word clean, canaries intact
    cache.close()
print("debug build ok")
"""


def test_debug_build_bounds_checks_and_canaries():
    from bit_asymmetric_kv_kvq_gb300 import _build
    lib = _build.build_debug()
    env = dict(os.environ, KVQ_LIB=lib)
    r = subprocess.run([sys.executable, "-c", _DEBUG_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout


def test_normal_build_has_no_debug_check():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    if kvq.kvq.LIB_PATH.endswith("libkvq_debug.so"):
        pytest.skip("running on the debug build")
    cache = kvq.KVCache.for_workload(CASES["mma"])
    assert kvq.kvq.kvq_debug_check(cache.handle) == kvq.kvq.KVQ_ERR_UNSUPPORTED
    cache.close()
