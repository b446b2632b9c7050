"""Host-side arithmetic of bench.py's decode legs (CPU): the bytes of one expert and of
the distinct experts a layer's routing touches, against hand counts
("Maple-Preview ...", section "The 5.31 GB claim reconciles": five trits per byte)."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_expert_bytes_at_the_maple_shape():
    # gate and up 512 x 410 B, down 2048 x 103 B, scales (512 + 512 + 2048) x 4 B
    assert bench.expert_bytes(2048, 512) == 2 * 512 * 410 + 2048 * 103 + 4 * 3072 == 643_072
    assert bench.expert_bytes(13, 7) == 2 * 7 * 3 + 13 * 2 + 4 * (14 + 13)


def test_distinct_expert_bytes_counts_each_layer_once_per_expert():
    one = bench.expert_bytes(16, 8)
    layer0 = torch.tensor([[3, 1], [1, 3], [3, 2]], dtype=torch.int32)  # experts {1, 2, 3}
    layer1 = torch.tensor([[0, 0], [-1, 9]], dtype=torch.int32)        # {0}; -1 and 9 are outside E = 4
    assert bench.distinct_expert_bytes([layer0, layer1], 4, 16, 8) == (3 + 1) * one
    assert bench.distinct_expert_bytes([], 4, 16, 8) == 0
