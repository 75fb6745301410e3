"""Test infrastructure: a plain model of the KV block allocator with one block
bitmap per (layer, KV head), the state management of the section on KDA
("国产AI芯片完成前沿大模型Day-0适配:稀疏注意力与混合精度推理全解析", §2.4: the
allocator allocates and reclaims KV cache blocks, knows the layer and the head,
and keeps an independent block bitmap per head so that heads do not overwrite
one another's blocks).  Only the tests import it; the library's allocator
(C++, kv_alloc.cpp) shares nothing with it.

Policy (not fixed by the article; the library's own): a request takes the
lowest free block ids of that (layer, head), in ascending order, or nothing if
fewer are free; a release must name blocks that (layer, head) holds, each once,
else it changes nothing.
"""


class BitmapKDA:
    def __init__(self, num_layers: int, num_heads: int, num_blocks: int):
        if num_layers < 1 or num_heads < 1 or num_blocks < 1:
            raise ValueError("sizes must be positive")
        self.num_blocks = num_blocks
        # in_use[layer][head] is the set of block ids that (layer, head) holds
        self.in_use = [[set() for _ in range(num_heads)] for _ in range(num_layers)]

    def alloc(self, layer: int, head: int, n: int):
        """The n lowest free ids of (layer, head), or None (nothing changes)."""
        held = self.in_use[layer][head]
        free = [i for i in range(self.num_blocks) if i not in held]
        if n < 0 or n > len(free):
            return None
        ids = free[:n]
        held.update(ids)
        return ids

    def free(self, layer: int, head: int, ids) -> bool:
        held = self.in_use[layer][head]
        ids = list(ids)
        if len(set(ids)) != len(ids) or any(i not in held for i in ids):
            return False
        held.difference_update(ids)
        return True

    def num_free(self, layer: int, head: int) -> int:
        return self.num_blocks - len(self.in_use[layer][head])

    def bitmap(self, layer: int, head: int) -> list:
        """The bitmap as 64-bit words, bit i of word i // 64 set when block i is held."""
        words = [0] * ((self.num_blocks + 63) // 64)
        for i in self.in_use[layer][head]:
            words[i // 64] |= 1 << (i % 64)
        return words
