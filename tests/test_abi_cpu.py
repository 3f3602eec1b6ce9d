"""The C ABI on a machine without a GPU: the library loads, exports every
function include/attn_varlen.h declares, and rejects bad arguments on the host
before touching a device."""
import ctypes

import pytest

import attention_attn_varlen_gb300 as av


@pytest.fixture(scope="module")
def L():
    av.build()
    return av.lib()


def test_every_declared_symbol_is_exported(L):
    names = av.exported_symbols()
    assert {"attn_varlen_fwd", "attn_decode_paged", "store_kvcache"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_status_strings(L):
    assert L.attn_abi_version() == 2
    for s in range(9):
        assert L.attn_status_string(s)
    assert L.attn_status_string(99) == b"unknown status"


def test_host_validation_without_device(L):
    null = None
    # store_kvcache: null pointers / negative sizes
    assert L.store_kvcache(null, null, null, null, null, null, 5, 8, 128, 0, 0, 10, null) == 1
    assert L.store_kvcache(null, null, null, null, null, null, -1, 8, 128, 0, 0, 10, null) == 1
    assert L.store_kvcache(null, null, null, null, null, null, 0, 8, 128, 0, 0, 10, null) == 0   # nothing to do
    # the failure-detection self-test needs somewhere to put its result
    assert L.attn_selftest_bounded_wait(null, null) == 1
    fake = ctypes.c_void_p(0x1000)
    # varlen: Hq not a multiple of Hkv, bad scale, unsupported head_dim, misaligned stride
    args = lambda **kw: [fake, fake, fake, fake, null, fake, fake, kw.get("B", 2), 8, 8, 4, 4, kw.get("Hq", 4),
                         kw.get("Hkv", 4), kw.get("D", 64), kw.get("scale", 0.125), 1, kw.get("bt", null), 0, 0, 0,
                         kw.get("v16", null), kw.get("qs", 0), 0, 0, 0, null, 0, null]
    assert L.attn_varlen_fwd(*args(Hq=6, Hkv=4)) == 1
    assert L.attn_varlen_fwd(*args(scale=0.0)) == 1
    assert L.attn_varlen_fwd(*args(scale=float("nan"))) == 1
    assert L.attn_varlen_fwd(*args(D=96)) == 2
    assert L.attn_varlen_fwd(*args(Hq=258, Hkv=2)) == 2      # a group of 129 heads exceeds the 128-row slot
    assert L.attn_varlen_fwd(*args(qs=4 * 64 + 3)) == 1        # row stride not 16-byte aligned
    assert L.attn_varlen_fwd(*args(B=0)) == 1
    assert L.attn_varlen_fwd(*args(v16=fake)) == 1            # a V / 16 cache needs a block table
    # decode: block size must be a power of two >= 16; group <= 64
    dec = lambda **kw: [fake, fake, fake, fake, null, fake, fake, 4, 2, kw.get("Hq", 8), kw.get("Hkv", 8), 128,
                        kw.get("bs", 16), 10, 64, 0.1, 0, 0, 0, null, 0, null]
    assert L.attn_decode_paged(*dec(bs=24)) == 1
    assert L.attn_decode_paged(*dec(Hq=128, Hkv=1)) == 2


def test_decode_split_rule_is_host_side(L):
    # no device: the rule falls back to a default SM count but stays well defined
    assert L.attn_decode_num_splits(256, 8, 16384, 0) == 4      # at most 4096 tokens per split
    assert L.attn_decode_num_splits(1, 8, 16384, 0) >= 8
    assert L.attn_decode_num_splits(4, 8, 100, 5) == 2          # capped by 64-token tiles
    assert L.attn_decode_workspace_size(256, 32, 8, 128, 16384, 1) == 0


def test_new_entries_validate_on_the_host(L):
    """kv-cache, padded and softmax entries reject bad arguments before any device work."""
    null = None
    fake = ctypes.c_void_p(0x1000)
    L.attn_kvcache_fwd.restype = ctypes.c_int
    L.attn_padded_fwd.restype = ctypes.c_int
    L.attn_softmax_rows.restype = ctypes.c_int
    # kv-cache: null pointers, non-positive seqlen_q, batch
    assert L.attn_kvcache_fwd(null, fake, fake, fake, null, fake, fake, 4, 2, 3, 32, 8, 128, 16, 64, 64,
                              ctypes.c_float(0.1), 1, null, fake, ctypes.c_size_t(1 << 30), null) == 1
    assert L.attn_kvcache_fwd(fake, fake, fake, fake, null, fake, fake, 4, 2, 0, 32, 8, 128, 16, 64, 64,
                              ctypes.c_float(0.1), 1, null, fake, ctypes.c_size_t(1 << 30), null) == 1
    # padded: null q, zero batch
    assert L.attn_padded_fwd(null, fake, fake, fake, null, null, null, 2, 16, 16, 8, 8, 64, ctypes.c_float(0.1), 1,
                             fake, ctypes.c_size_t(1 << 30), null) == 1
    assert L.attn_padded_fwd(fake, fake, fake, fake, null, null, null, 0, 16, 16, 8, 8, 64, ctypes.c_float(0.1), 1,
                             fake, ctypes.c_size_t(1 << 30), null) == 1
    # softmax: null pointers, negative rows, unknown dtype, stride shorter than a row
    i64 = ctypes.c_int64
    assert L.attn_softmax_rows(null, fake, i64(4), 8, i64(0), i64(0), 0, null) == 1
    assert L.attn_softmax_rows(fake, fake, i64(-1), 8, i64(0), i64(0), 0, null) == 1
    assert L.attn_softmax_rows(fake, fake, i64(4), 8, i64(0), i64(0), 7, null) == 1
    assert L.attn_softmax_rows(fake, fake, i64(4), 8, i64(4), i64(0), 0, null) == 1


def test_new_workspace_sizes_are_host_side(L):
    L.attn_kvcache_workspace_size.restype = ctypes.c_size_t
    L.attn_padded_workspace_size.restype = ctypes.c_size_t
    assert L.attn_kvcache_workspace_size(0, 1, 32, 8, 128, 100) == 0
    assert L.attn_padded_workspace_size(2, 0, 16, 8, 8, 64) == 0
    a = L.attn_kvcache_workspace_size(4, 40, 32, 8, 128, 1000)
    b = L.attn_kvcache_workspace_size(4, 40, 32, 8, 128, 2000)
    assert 0 < a < b            # two-slot prefill route (40 x 4 query rows per KV head): the fp16 V' copy grows with the cache
    # one-slot prefill route at head_dim 128 (17 x 4 rows): V tiles are converted in the kernel, no V' copy
    assert 0 < L.attn_kvcache_workspace_size(4, 17, 32, 8, 128, 1000) == L.attn_kvcache_workspace_size(4, 17, 32, 8, 128, 1 << 20)
    L.attn_varlen_workspace_size.restype = ctypes.c_size_t
    i64 = ctypes.c_int64
    assert L.attn_varlen_workspace_size(4, 32, 8, 128, 32, i64(1000)) == L.attn_varlen_workspace_size(4, 32, 8, 128, 32, i64(10 ** 7))
    assert L.attn_varlen_workspace_size(4, 32, 8, 128, 33, i64(1000)) < L.attn_varlen_workspace_size(4, 32, 8, 128, 33, i64(10 ** 7))
    assert L.attn_varlen_workspace_size(4, 32, 8, 64, 32, i64(1000)) < L.attn_varlen_workspace_size(4, 32, 8, 64, 32, i64(10 ** 7))
    # decode route (3 x 4 rows): only split partials, at most 64 splits of fp32 rows, whatever the cache length
    for n in (0, 1000, 1 << 20):
        c = L.attn_kvcache_workspace_size(4, 3, 32, 8, 128, n)
        assert 0 < c <= 4 * 3 * 32 * 64 * 129 * 4 + 256
    assert L.attn_padded_workspace_size(2, 16, 64, 8, 8, 64) > 0


def test_host_entry_checks_offsets_on_the_host(L):
    """attn_varlen_fwd_host reads cu_seqlens in host memory and refuses offsets
    that do not start at 0, decrease, or exceed the stated maxima, before it
    queries a device or queues a copy."""
    null = None
    fake = ctypes.c_void_p(0x1000)

    def cu(*v):
        a = (ctypes.c_int32 * len(v))(*v)
        return a, ctypes.cast(a, ctypes.c_void_p)

    keep = []

    def call(cq, ck, mq=100, mk=100, groups=4, ev=fake):
        (aq, pq), (ak, pk) = cu(*cq), cu(*ck)
        keep.extend([aq, ak])
        return L.attn_varlen_fwd_host(fake, fake, fake, fake, pq, pk, len(cq) - 1, mq, mk, 8, 2, 64,
                                      ctypes.c_float(0.125), 1, fake, fake, fake, fake, fake, fake,
                                      ctypes.c_size_t(1 << 20), groups, null, null, null, ev, ev)

    assert call([0, 120, 150], [0, 100, 150]) == 1      # a query length above max_seqlen_q
    assert call([1, 100, 150], [0, 100, 150]) == 1      # does not start at 0
    assert call([0, 100, 90], [0, 100, 150]) == 1       # decreasing
    assert call([0, 100, 150], [0, 100, 250]) == 1      # a key length above max_seqlen_k
    assert call([0, 100, 150], [0, 100, 150], groups=0) == 1
    assert call([0, 100, 150], [0, 100, 150], ev=null) == 1
    # valid offsets reach the device query, which fails without a GPU
    assert call([0, 100, 150], [0, 100, 150]) == 7


def test_group_sizes_that_do_not_divide_128(L):
    """Prefill sizes for any group up to 128 heads per KV head: floor(128 / G) tokens
    per slot, so the unit list grows with ceil(Lq / (2 floor(128 / G))); G > 128 is
    refused (size 0)."""
    L.attn_varlen_workspace_size.restype = ctypes.c_size_t
    i64 = ctypes.c_int64
    # head_dim 64 (no one-slot instance): header + V' copy + unit list
    for G, tps in ((3, 42), (5, 25), (6, 21), (7, 18), (48, 2), (96, 1), (128, 1)):
        one = L.attn_varlen_workspace_size(2, G, 1, 64, 2 * tps, i64(0))
        two = L.attn_varlen_workspace_size(2, G, 1, 64, 2 * tps + 1, i64(0))
        assert 0 < one < two, G   # one more query pair per sequence past 2 floor(128 / G) tokens
    assert L.attn_varlen_workspace_size(2, 129, 1, 64, 8, i64(0)) == 0
    # the kv-cache entry: G = 5 at head_dim 128, 8 new tokens = 40 rows -> one-slot prefill,
    # no V' copy; 3 new tokens = 15 rows -> decode partials only
    L.attn_kvcache_workspace_size.restype = ctypes.c_size_t
    assert L.attn_kvcache_workspace_size(4, 8, 40, 8, 128, 1000) == L.attn_kvcache_workspace_size(4, 8, 40, 8, 128, 10 ** 6)
    assert 0 < L.attn_kvcache_workspace_size(4, 3, 40, 8, 128, 10 ** 6) <= 4 * 3 * 40 * 64 * 129 * 4 + 256
