"""Host-side logic with no GPU: the bench's launch count and super-batch
bookkeeping, and the huge-page check of the host-table allocator."""
import mmap

import numpy as np
import torch

import bench
from sampling_gnn_mini_gb300 import hostmem


def test_kernels_per_step_matches_the_launch_lists():
    # counts seen in ncu launch lists and bench lines on GB300: Mid 24, Tiny 19,
    # Skew (super-batch of 8) 20, Billion with region-ordered misses 30, Wide 25
    assert bench.kernels_per_step(3, 1) == 24
    assert bench.kernels_per_step(2, 1) == 19
    assert bench.kernels_per_step(2, 8) == 20
    assert bench.kernels_per_step(3, 1, by_region=True) == 30
    assert bench.kernels_per_step(2, 1, by_region=True) == 25
    assert bench.kernels_per_step(1, 1) == 2 + 3 + 5 + 1 + 1 + 1  # one hop: a single gather call


def _super_counts(per_sub, H):
    """counts as the sampler writes them: totals, then (2H+1) entries per
    mini-batch (node counts per hop, then edge counts)."""
    c = np.zeros((2 * H + 1) * (1 + len(per_sub)), np.int64)
    for k, (nodes, edges) in enumerate(per_sub):
        base = (2 * H + 1) * (1 + k)
        c[base: base + H + 1] = nodes
        c[base + H + 1: base + 2 * H + 1] = edges
        c[: H + 1] += nodes
        c[H + 1: 2 * H + 1] += edges
    return c


def test_frontier_ids_of_a_super_batch():
    H = 2
    # mini-batch 0: V_0 = {5, 6}, V_1 adds 7, V_2 adds 8, 9
    # mini-batch 1: V_0 = {7, 1}, V_1 adds 5, V_2 adds 2
    unique = np.array([5, 6, 7, 8, 9, 7, 1, 5, 2], np.int32)
    counts = _super_counts([([2, 3, 5], [3, 4]), ([2, 3, 4], [2, 2])], H)
    assert counts[H] == len(unique)
    assert bench.frontier_ids(counts, unique, H, 2, 0).tolist() == [1, 5, 6, 7]
    assert bench.frontier_ids(counts, unique, H, 2, 1).tolist() == [1, 5, 6, 7]
    assert bench.frontier_ids(counts, unique, H, 2, 2).tolist() == [1, 2, 5, 6, 7, 8, 9]
    # one mini-batch: the prefix of unique
    c1 = _super_counts([([2, 3, 5], [3, 4])], H)[: 2 * H + 1]
    assert bench.frontier_ids(c1, unique[:5], H, 1, 1).tolist() == [5, 6, 7]


def test_huge_page_bytes_from_smaps():
    lines = ["7f0000000000-7f0040000000 rw-p 00000000 00:00 0 \n",
             "Size:            1048576 kB\n",
             "AnonHugePages:    524288 kB\n",
             "7f0040000000-7f0080000000 rw-p 00000000 00:00 0 \n",
             "Size:            1048576 kB\n",
             "AnonHugePages:         0 kB\n",
             "VmFlags: rd wr mr mw me ac\n"]
    assert hostmem.huge_bytes_in(0x7F0000000000, lines) == 524288 * 1024
    assert hostmem.huge_bytes_in(0x7F0040000000, lines) == 0
    assert hostmem.huge_bytes_in(0x123000, lines) == 0
    # this process's own mapping: a value within the mapping's size
    n = 64 << 20
    m = mmap.mmap(-1, n, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    if hasattr(mmap, "MADV_HUGEPAGE"):
        m.madvise(mmap.MADV_HUGEPAGE)
    t = torch.frombuffer(m, dtype=torch.uint8)
    t.fill_(1)
    assert 0 <= hostmem._huge_bytes(t.data_ptr()) <= n
    del t


def test_lock_pages_locks_a_mapping_or_reports_refusal():
    # mlock of a small mapping: True where the process may lock memory (as root
    # here), and a plain False, never an exception, where it is refused; the
    # mapping stays readable and writable either way, and a locked one shows
    # up in the process's locked total
    n = 4 << 20
    m = mmap.mmap(-1, n, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    t = torch.frombuffer(m, dtype=torch.uint8)
    t.fill_(3)

    def vm_lck_kb():
        with open("/proc/self/status") as fh:
            for line in fh:
                if line.startswith("VmLck:"):
                    return int(line.split()[1])
        return 0

    before = vm_lck_kb()
    ok = hostmem._lock_pages(t.data_ptr(), n)
    assert isinstance(ok, bool)
    if ok:
        assert vm_lck_kb() - before >= n // 1024
    t[::4096] += 1
    assert int(t[4096]) == 4 and int(t[1]) == 3
    assert hostmem._lock_pages(0, 0) in (True, False)
    del t
    m.close()
