"""GPU parity of the KV4 cache and its decode attention.

* qoq_kv4_append: every slot it writes, decoded by a numpy reader written
  from the page-format text in include/qoq.h, holds the oracle's codes,
  scale and zero bit for bit; slots it does not own keep their fill bytes.
* qoq_kv4_decode_attention: against the oracle's fp64 attention over the
  oracle's own quantized keys and values, per (sequence, query head) row:
  |O - O_ref| <= 2e-3 * max_d |O_ref| + ulp16(|O_ref|), for grouped-query
  ratios 1, 2, 4 and 8, ragged lengths (page tails), split sequences, empty
  sequences, many short sequences, a single token, repeated calls on one
  workspace, and the Llama-3-8B decode workload (batch 64, lengths 512-1536).
"""
import numpy as np
import pytest

import oracle
import w4a8_quantized_serving_qoq_gb300 as qoq

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128
PT = 64
CHUNK = 8704
FILL = 0xEE


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


# ---- the page format, read as the header states it ----
def _nibble_dims():
    kd = np.zeros((16, 8), np.int64)
    vd = np.zeros((16, 8), np.int64)
    for i in range(16):
        for j in range(8):
            r, jj = divmod(i, 4)
            a, b = j & 3, j >> 2
            kd[i, j] = 32 * jj + 16 * (a & 1) + 8 * (a >> 1) + 2 * r + b
            g, w = divmod(i, 2)
            vd[i, j] = g + 8 * (8 * w + j)
    return kd, vd


KDIMS, VDIMS = _nibble_dims()


def read_slot(pages, page, h, slot, which):
    """(codes [128], s bits, z bits) of one slot; which = 0 keys, 1 values."""
    chunk = pages[page, h * CHUNK:(h + 1) * CHUNK]
    base = 0 if which == 0 else 4096 + 256
    words = chunk[base + 64 * slot: base + 64 * slot + 64].view("<u4")
    nib = (words[:, None] >> (4 * np.arange(8, dtype=np.uint32))[None, :]) & 15
    codes = np.zeros(D, np.uint8)
    codes[(KDIMS if which == 0 else VDIMS).reshape(-1)] = nib.reshape(-1)
    meta = int(chunk[base + 4096 + 4 * slot: base + 4096 + 4 * slot + 4].view("<u4")[0])
    return codes, meta & 0xFFFF, meta >> 16


# ---- a synthetic cache ----
def make_cache(lens, hkv, seed, extra_pages=3):
    """Keys with fixed outlier channels per head (x10, as the pages observe for
    the key cache), plain N(0,1) values; every sequence's pages drawn at random
    from one pool."""
    rng = np.random.default_rng(seed)
    max_pages = max(1, max((L + PT - 1) // PT for L in lens))
    npages = [(L + PT - 1) // PT for L in lens]
    num_pages = sum(npages) + extra_pages
    perm = rng.permutation(num_pages)
    table = np.full((len(lens), max_pages), -1, np.int32)
    k = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[k:k + n]
        k += n
    T = sum(lens)
    K = rng.standard_normal((T, hkv, D)).astype(np.float32)
    for h in range(hkv):
        K[:, h, rng.choice(D, 3, replace=False)] *= 10.0
    V = rng.standard_normal((T, hkv, D)).astype(np.float32)
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)]) if T else np.zeros(0, np.int32)
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens]) if T else np.zeros(0, np.int32)
    return dict(K=K.astype(np.float16), V=V.astype(np.float16), seq=seq, pos=pos, table=table,
                num_pages=num_pages, max_pages=max_pages, lens=np.array(lens, np.int32))


def device_pages(c, hkv, order=None):
    pages = torch.full((c["num_pages"], qoq.qoq_kv4_page_bytes(hkv)), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    idx = np.arange(len(c["seq"])) if order is None else order
    if len(idx):
        qoq.qoq_kv4_append(_t(c["K"][idx]), _t(c["V"][idx]), _t(c["seq"][idx]), _t(c["pos"][idx]), _t(c["table"]),
                           pages, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return pages


def test_append_writes_the_oracle_codes_in_the_page_format():
    hkv = 3
    c = make_cache([5, 64, 130], hkv, 11)
    order = np.random.default_rng(1).permutation(len(c["seq"]))  # tokens in any order
    pages = device_pages(c, hkv, order).cpu().numpy()
    qk, sk, zk = oracle.kv4_quantize(c["K"].reshape(-1, D))
    qv, sv, zv = oracle.kv4_quantize(c["V"].reshape(-1, D))
    owned = set()
    for t in range(len(c["seq"])):
        b, p = c["seq"][t], c["pos"][t]
        page, slot = c["table"][b, p // PT], p % PT
        for h in range(hkv):
            i = t * hkv + h
            codes, s, z = read_slot(pages, page, h, slot, 0)
            assert np.array_equal(codes, qk[i]) and s == sk.view(np.uint16)[i] and z == zk.view(np.uint16)[i]
            codes, s, z = read_slot(pages, page, h, slot, 1)
            assert np.array_equal(codes, qv[i]) and s == sv.view(np.uint16)[i] and z == zv.view(np.uint16)[i]
            owned.add((page, h, slot))
    # every byte of a slot nobody owns still holds the fill pattern
    for page in range(c["num_pages"]):
        for h in range(hkv):
            chunk = pages[page, h * CHUNK:(h + 1) * CHUNK]
            for slot in range(PT):
                if (page, h, slot) in owned:
                    continue
                for base in (0, 4352):
                    assert (chunk[base + 64 * slot: base + 64 * slot + 64] == FILL).all()
                    assert (chunk[base + 4096 + 4 * slot: base + 4096 + 4 * slot + 4] == FILL).all()


def test_append_skips_out_of_range_tokens_and_reports_them():
    c = make_cache([10], 1, 12)
    pages = torch.full((c["num_pages"], qoq.qoq_kv4_page_bytes(1)), FILL, dtype=torch.uint8, device=DEV)
    status = torch.zeros((1,), dtype=torch.int32, device=DEV)
    seq = c["seq"].copy()
    pos = c["pos"].copy()
    seq[3] = 5            # no such sequence
    pos[4] = 64 * 9       # beyond the page table row
    table = c["table"].copy()
    qoq.qoq_kv4_append(_t(c["K"]), _t(c["V"]), _t(seq), _t(pos), _t(table), pages, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4
    host = pages.cpu().numpy()
    qk, _, _ = oracle.kv4_quantize(c["K"].reshape(-1, D))
    codes, _, _ = read_slot(host, table[0, 0], 0, 2, 0)
    assert np.array_equal(codes, qk[2])                          # a good token still lands
    assert (host[table[0, 0], 64 * 3: 64 * 5] == FILL).all()     # slots 3 and 4 untouched


def _reference(c, Q, hkv, scale):
    """Oracle attention per (sequence, KV head) on the oracle's quantized cache."""
    B, hq = Q.shape[0], Q.shape[1]
    G = hq // hkv
    T = len(c["seq"])
    qk, sk, zk = oracle.kv4_quantize(c["K"].reshape(-1, D))
    qv, sv, zv = oracle.kv4_quantize(c["V"].reshape(-1, D))
    qk, qv = qk.reshape(T, hkv, D), qv.reshape(T, hkv, D)
    sk, zk, sv, zv = (a.reshape(T, hkv) for a in (sk, zk, sv, zv))
    O = np.zeros((B, hq, D))
    start = 0
    for b, L in enumerate(c["lens"]):
        for h in range(hkv):
            if L == 0:
                continue
            sl = slice(start, start + L)
            O[b, h * G:(h + 1) * G] = oracle.kv4_attention_f64(
                Q[b, h * G:(h + 1) * G], qk[sl, h], sk[sl, h], zk[sl, h], qv[sl, h], sv[sl, h], zv[sl, h], scale)
        start += L
    return O


def _check(c, hkv, hq, seed):
    B = len(c["lens"])
    Q = np.random.default_rng(seed).standard_normal((B, hq, D)).astype(np.float16)
    scale = 1.0 / np.sqrt(D)
    pages = device_pages(c, hkv)
    ws = qoq.new_workspace(qoq.qoq_kv4_attention_workspace_bytes(B, hq, hkv, c["max_pages"]))
    O = qoq.qoq_kv4_decode_attention(_t(Q), pages, _t(c["table"]), _t(c["lens"]), hkv, scale, workspace=ws)
    torch.cuda.synchronize()
    assert qoq.qoq_workspace_status(ws)[0] == 0
    got = O.cpu().numpy().astype(np.float64).reshape(B * hq, D)
    ref = _reference(c, Q, hkv, scale).reshape(B * hq, D)
    ok = oracle.o_within_tolerance(got, ref)
    assert ok.all(), f"{int((~ok).sum())} outputs outside tolerance; worst {np.abs(got - ref).max()}"
    return got, ref


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_attention_matches_oracle_gqa_ratios(G):
    hkv = 2
    c = make_cache([1, 17, 64, 65, 300], hkv, 20 + G)
    _check(c, hkv, hkv * G, 30 + G)


@pytest.mark.parametrize("lens", [[4096], [3000, 5], [0, 129, 0]])
def test_attention_split_sequences_and_empty_ones(lens):
    """Few sequences with long contexts split across CTAs (merged by the
    second kernel); a sequence of length 0 gives zeros."""
    hkv, hq = 8, 32
    c = make_cache(lens, hkv, 40 + len(lens))
    got, _ = _check(c, hkv, hq, 41)
    for b, L in enumerate(lens):
        if L == 0:
            assert not got.reshape(len(lens), hq, D)[b].any()


def test_attention_llama3_8b_decode_batch():
    """The decode workload of the benchmark: 64 sequences, lengths drawn
    uniformly from 512..1536, 32 query heads over 8 KV heads."""
    lens = list(np.random.default_rng(50).integers(512, 1537, 64))
    hkv, hq = 8, 32
    c = make_cache(lens, hkv, 51)
    _check(c, hkv, hq, 52)


def test_attention_reports_bad_page_indices():
    hkv, hq = 1, 4
    c = make_cache([100], hkv, 60)
    pages = device_pages(c, hkv)
    table = c["table"].copy()
    table[0, 1] = c["num_pages"] + 7      # out of the pool: skipped, reported
    Q = np.ones((1, hq, D), np.float16)
    ws = qoq.new_workspace(qoq.qoq_kv4_attention_workspace_bytes(1, hq, hkv, c["max_pages"]))
    qoq.qoq_kv4_decode_attention(_t(Q), pages, _t(table), _t(c["lens"]), hkv, 0.088, workspace=ws)
    st, bits = qoq.qoq_workspace_status(ws)
    assert st == 7 and bits & 4


def test_attention_many_short_sequences():
    """700 sequences of 1 to 3 pages (more (sequence, KV head) pairs than
    resident CTAs), one of them empty."""
    lens = list(np.random.default_rng(70).integers(1, 193, 700))
    lens[5] = 0
    hkv, hq = 2, 8
    c = make_cache(lens, hkv, 71)
    got, _ = _check(c, hkv, hq, 72)
    assert not got.reshape(len(lens), hq, D)[5].any()


def test_attention_single_token():
    hkv, hq = 1, 4
    c = make_cache([1], hkv, 73)
    _check(c, hkv, hq, 74)


def test_attention_repeated_calls_reuse_the_workspace():
    """The same workspace gives the same outputs call after call, across
    shapes (split and unsplit sequences)."""
    hkv, hq = 8, 32
    c = make_cache([2000, 7, 900], hkv, 75)
    B = 3
    Q = np.random.default_rng(76).standard_normal((B, hq, D)).astype(np.float16)
    pages = device_pages(c, hkv)
    ws = qoq.new_workspace(qoq.qoq_kv4_attention_workspace_bytes(B, hq, hkv, c["max_pages"]))
    ref = _reference(c, Q, hkv, 0.05).reshape(B * hq, D)
    for _ in range(3):
        O = qoq.qoq_kv4_decode_attention(_t(Q), pages, _t(c["table"]), _t(c["lens"]), hkv, 0.05, workspace=ws)
        got = O.cpu().numpy().astype(np.float64).reshape(B * hq, D)
        assert oracle.o_within_tolerance(got, ref).all()
    c1 = make_cache([100], hkv, 77)
    Q1 = np.random.default_rng(78).standard_normal((1, hq, D)).astype(np.float16)
    O1 = qoq.qoq_kv4_decode_attention(_t(Q1), device_pages(c1, hkv), _t(c1["table"]), _t(c1["lens"]), hkv, 0.05,
                                      workspace=ws)
    assert oracle.o_within_tolerance(O1.cpu().numpy().astype(np.float64).reshape(hq, D),
                                     _reference(c1, Q1, hkv, 0.05).reshape(hq, D)).all()
    assert qoq.qoq_workspace_status(ws)[0] == 0
