"""Host-side parts of bench.py that run without a GPU: the replica time reduction across ranks (gloo,
two processes on CPU) and the reference arm (the fp64 oracle on a bounded sample of the workload)."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(1.5 + rank, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_replica_time_is_the_max_over_two_gloo_ranks():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_reference_arm_prints_its_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "ms" and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


class _FakeLib:
    """Stands in for the binding in split_pieces: records what each piece's bucket array would hold."""
    MUON_BF16 = 1

    def make_buckets(self, specs):
        return specs

    def pointer_array(self, tensors, device):
        return list(tensors)


class _Grads(list):
    def element_size(self):
        return 2


def _pieces_of(shapes, max_bytes=1.5e9):
    sys.path.insert(0, ROOT)
    import bench
    w = bench.Workload.__new__(bench.Workload)
    w.L, w.device = _FakeLib(), "cpu"
    w.buckets = [{"K": K, "A": A, "B": B, "g": _Grads(range(K)), "p": list(range(K)), "mom": list(range(K))}
                 for K, A, B in shapes]
    order, adamw_at = w.split_pieces(max_bytes)
    return w, order, adamw_at


def test_end_to_end_pieces_cover_every_matrix_once_in_the_pipeline_order():
    shapes = [(64, 4096, 4096), (64, 1024, 4096), (64, 14336, 4096), (32, 4096, 14336)]
    w, order, adamw_at = _pieces_of(shapes)
    seen = sorted((b, k) for b, k0, k1 in order for k in range(k0, k1))
    assert seen == sorted((b, k) for b, (K, _, _) in enumerate(shapes) for k in range(K))
    grad_bytes = lambda pc: (pc[2] - pc[1]) * shapes[pc[0]][1] * shapes[pc[0]][2] * 2
    assert all(grad_bytes(pc) <= 1.5e9 for pc in order)
    # the smallest bucket (1024x4096, one piece) in two halves first, AdamW after the next piece
    assert order[:2] == [(1, 0, 32), (1, 32, 64)] and adamw_at == 3
    # the largest piece last, in parts that halve down to one matrix
    tail = order[-4:]
    assert [k1 - k0 for _, k0, k1 in tail] == [6, 3, 1, 1] and len({b for b, _, _ in tail}) == 1
    assert all(tail[i][2] == tail[i + 1][1] for i in range(3))
    # each piece's bucket array holds exactly its matrices
    for (b, k0, k1), arr in zip(order, w.piece_arrays):
        (params, grads, mom, K, A, B, _, _), = arr
        assert params == list(range(k0, k1)) and grads == list(range(k0, k1)) and K == k1 - k0
        assert (A, B) == shapes[b][1:]


@pytest.mark.parametrize("shapes", [[(1, 64, 128)], [(3, 64, 128), (1, 32, 32)], [(2, 8, 8), (2, 8, 8)]])
def test_end_to_end_pieces_of_small_sets(shapes):
    _, order, adamw_at = _pieces_of(shapes)
    seen = sorted((b, k) for b, k0, k1 in order for k in range(k0, k1))
    assert seen == sorted((b, k) for b, (K, _, _) in enumerate(shapes) for k in range(K))
    assert all(k1 > k0 for _, k0, k1 in order) and 1 <= adamw_at <= len(order)
