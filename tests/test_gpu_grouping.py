"""Grouping of token slots by expert (the permute step), through moe_group_by_expert.

The grouping is stable, so its result is unique: counts are the histogram of the
ids, offsets its exclusive prefix sum, and perm the slot indices sorted by expert
with ties in slot order -- exactly numpy's stable argsort of the flattened ids.
Cases cover the one-CTA form (up to 2048 slots) and the multi-CTA form (several
chunks of 2048 slots), hot experts, idle experts, the largest E, and ids outside
[0, E), which are flagged and left out.
"""
import numpy as np
import pytest

from gpu_util import moe_lib, need_gpu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

CASES = [  # (T, k, E, kind)
    (1, 1, 1, "uniform"),
    (7, 3, 8, "uniform"),
    (64, 8, 256, "uniform"),          # 512 slots: the one-CTA form
    (256, 8, 256, "uniform"),         # exactly 2048 slots
    (257, 8, 256, "uniform"),         # 2056 slots: two chunks
    (4096, 8, 256, "skewed"),         # 32768 slots, 16 chunks, hot experts
    (8192, 4, 32, "skewed"),
    (3000, 2, 1024, "uniform"),       # the largest E
    (5000, 4, 16, "one-hot"),         # every slot to two experts: long runs across chunks
]


def _ids(T, k, E, kind, rng):
    if kind == "uniform":
        return np.stack([rng.permutation(E)[:k] if k <= E else rng.integers(0, E, k) for _ in range(T)])
    if kind == "skewed":
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    ids = np.zeros((T, k), np.int64)
    ids[:, 0] = 3
    ids[:, 1:] = 11
    return ids


@pytest.mark.parametrize("T,k,E,kind", CASES, ids=lambda v: str(v))
def test_grouping_is_the_stable_sort(T, k, E, kind):
    need_gpu()
    moe = moe_lib()
    rng = np.random.default_rng(T * 131 + k * 7 + E)
    ids = _ids(T, k, E, kind, rng).astype(np.int32)
    cfg = moe.qwen_cfg(d_model=64, n_experts=E, top_k=k, expert_ff=32, shared_ff=0)
    ws = moe.workspace(cfg, T)
    ws.fill_(0xAB)
    counts, offsets, perm = moe.moe_group_by_expert(cfg, torch.from_numpy(ids).cuda(), ws=ws)
    assert moe.moe_device_status(ws)[0] == 0
    flat = ids.reshape(-1)
    want_counts = np.bincount(flat, minlength=E)
    assert np.array_equal(counts.cpu().numpy(), want_counts)
    assert np.array_equal(offsets.cpu().numpy(), np.concatenate([[0], np.cumsum(want_counts)]))
    assert np.array_equal(perm.cpu().numpy()[:T * k], np.argsort(flat, kind="stable"))


def test_bad_ids_are_left_out_and_flagged():
    need_gpu()
    moe = moe_lib()
    T, k, E = 300, 3, 16
    rng = np.random.default_rng(5)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[4, 1] = E
    ids[17, 0] = -1
    ids[299, 2] = 1 << 20
    cfg = moe.qwen_cfg(d_model=64, n_experts=E, top_k=k, expert_ff=32, shared_ff=0)
    ws = moe.workspace(cfg, T)
    counts, offsets, perm = moe.moe_group_by_expert(cfg, torch.from_numpy(ids).cuda(), ws=ws)
    st, bits = moe.moe_device_status(ws)
    assert st == -6 and bits & 1
    flat = ids.reshape(-1)
    good = (flat >= 0) & (flat < E)
    assert np.array_equal(counts.cpu().numpy(), np.bincount(flat[good], minlength=E))
    n = int(good.sum())
    assert int(offsets[E]) == n
    order = np.nonzero(good)[0][np.argsort(flat[good], kind="stable")]
    assert np.array_equal(perm.cpu().numpy()[:n], order)


def test_zero_tokens():
    need_gpu()
    moe = moe_lib()
    cfg = moe.qwen_cfg(d_model=64, n_experts=8, top_k=2, expert_ff=32, shared_ff=0)
    counts, offsets, _ = moe.moe_group_by_expert(cfg, torch.empty((0, 2), dtype=torch.int32, device="cuda"))
    assert counts.cpu().tolist() == [0] * 8 and offsets.cpu().tolist() == [0] * 9
