"""Radix prefix cache, the oracle's version (test infrastructure only).

A plain restatement of "KV Cache Management" (cs249r vol. 3 ch. 5), "Prefix Caching
Across Turns", on top of the oracle's block pool:

* Table 4 node layout: prefix_tokens, block_ids, children (keyed by the branch), parent,
  ref_count, last_access.  Definition 0.2: a radix tree indexing physical blocks by tokens.
* "Longest prefix matching": the walk from the root consumes edge slices that match the
  prompt; only fully packed blocks are shared, so the usable match is rounded down to
  whole blocks.  Read here as a tree over whole blocks: an edge holds whole blocks and the
  child map is keyed by the child's first block (the B tokens after the branch point).
* "Dynamic radix eviction", steps 1-4: pinned (ref_count >= 1) vs dormant nodes, an LRU
  queue of dormant leaves by last_access, pop the oldest and release all its blocks while
  free blocks are below the target, a parent left childless and dormant joins the queue.
* Eq. 2: hit rate = sum of matched tokens / sum of prompt tokens.

Conventions shared with the library's C ABI (its header states them): one clock tick per
attach / insert / release, stamping every node the operation traverses; LRU ties go to
the node created first; a node matched or inserted only in part is split at that block
boundary, the new upper node taking the earlier blocks, the parent's reference count and
stamp; the cache holds one owner reference on each block it indexes.

Pure Python loops: small cases only.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple


class Node:
    def __init__(self, parent: Optional["Node"], serial: int):
        self.prefix_tokens: List[int] = []
        self.block_ids: List[int] = []
        self.children: Dict[Tuple[int, ...], "Node"] = {}
        self.parent = parent
        self.ref_count = 0
        self.last_access = 0
        self.serial = serial


class RadixCache:
    def __init__(self, pool, block_size: int):
        self.pool = pool  # oracle.Pool
        self.B = block_size
        self.root = Node(None, 0)
        self.clock = 0
        self.serial = 0
        self.pins: Dict[int, Node] = {}  # request (sequence id) -> deepest matched node
        self.prompt_tokens = 0
        self.matched_tokens = 0

    # -- helpers ------------------------------------------------------------------
    def _new_node(self, parent: Optional[Node]) -> Node:
        self.serial += 1
        return Node(parent, self.serial)

    def _blocks_of(self, tokens: List[int]) -> List[Tuple[int, ...]]:
        B = self.B
        return [tuple(tokens[i * B:(i + 1) * B]) for i in range(len(tokens) // B)]

    def _edge_blocks(self, node: Node) -> List[Tuple[int, ...]]:
        return self._blocks_of(node.prefix_tokens)

    def _split(self, node: Node, k: int) -> Node:
        """The first k blocks of `node` become a new node between it and its parent."""
        parent = node.parent
        key = tuple(node.prefix_tokens[:self.B])
        del parent.children[key]
        upper = self._new_node(parent)
        upper.prefix_tokens = node.prefix_tokens[:k * self.B]
        upper.block_ids = node.block_ids[:k]
        upper.ref_count = node.ref_count
        upper.last_access = node.last_access
        node.prefix_tokens = node.prefix_tokens[k * self.B:]
        node.block_ids = node.block_ids[k:]
        node.parent = upper
        upper.children[tuple(node.prefix_tokens[:self.B])] = node
        parent.children[key] = upper
        return upper

    def _walk(self, prompt_blocks):
        """(deepest fully matched node, partly matched child or None, its matched blocks, total)."""
        node, i = self.root, 0
        while i < len(prompt_blocks):
            child = node.children.get(prompt_blocks[i])
            if child is None:
                break
            edge = self._edge_blocks(child)
            j = 0
            while j < len(edge) and i + j < len(prompt_blocks) and edge[j] == prompt_blocks[i + j]:
                j += 1
            i += j
            if j < len(edge):
                return node, child, j, i
            node = child
        return node, None, 0, i

    def _path_blocks(self, node: Node) -> List[int]:
        path = []
        while node is not None and node.parent is not None:
            path.append(node)
            node = node.parent
        out = []
        for n in reversed(path):
            out += n.block_ids
        return out

    # -- operations ---------------------------------------------------------------
    def match(self, tokens: List[int]) -> Tuple[int, List[int]]:
        """Longest whole-block prefix: (matched tokens, its blocks)."""
        node, part, k, total = self._walk(self._blocks_of(tokens))
        blocks = self._path_blocks(node) + (part.block_ids[:k] if part is not None else [])
        return total * self.B, blocks

    def attach(self, tokens: List[int]) -> Tuple[int, int]:
        """Serve a request: (new sequence id, matched tokens)."""
        node, part, k, total = self._walk(self._blocks_of(tokens))
        deepest = self._split(part, k) if part is not None else node
        blocks = self._path_blocks(deepest)
        seq = self.pool.seq_adopt(blocks, total * self.B)
        self.clock += 1
        n = deepest
        while n is not self.root:
            n.ref_count += 1
            n.last_access = self.clock
            n = n.parent
        self.pins[seq] = deepest
        self.prompt_tokens += len(tokens)
        self.matched_tokens += total * self.B
        return seq, total * self.B

    def insert(self, seq: int, tokens: List[int]) -> None:
        """Index the sequence's whole blocks under its tokens."""
        table = [int(x) for x in self.pool.table(seq)]
        assert len(tokens) <= self.pool.seq_len(seq)
        blocks = self._blocks_of(tokens)
        self.clock += 1
        node, i = self.root, 0
        while i < len(blocks):
            child = node.children.get(blocks[i])
            if child is None:
                leaf = self._new_node(node)
                leaf.prefix_tokens = [t for b in blocks[i:] for t in b]
                leaf.block_ids = table[i:len(blocks)]
                for p in leaf.block_ids:
                    self.pool.block_retain(p)
                leaf.last_access = self.clock
                node.children[blocks[i]] = leaf
                break
            edge = self._edge_blocks(child)
            j = 0
            while j < len(edge) and i + j < len(blocks) and edge[j] == blocks[i + j]:
                j += 1
            if j < len(edge):
                child = self._split(child, j)
            child.last_access = self.clock
            node = child
            i += j

    def release(self, seq: int) -> None:
        deepest = self.pins.pop(seq)
        self.clock += 1
        n = deepest
        while n is not self.root:
            n.ref_count -= 1
            n.last_access = self.clock
            n = n.parent

    def _nodes(self):
        stack = [self.root]
        while stack:
            n = stack.pop()
            for c in n.children.values():
                yield c
                stack.append(c)

    def evict(self, target_free: int) -> int:
        """Leaf-first LRU eviction until the pool holds target_free free blocks."""
        # 1-2: the dormant leaves, ordered by last access (then creation)
        queue = [n for n in self._nodes() if n.ref_count == 0 and not n.children]
        released = 0
        # 3: pop the least recently used leaf, release its blocks, unlink it
        while len(self.pool.free_list()) < target_free and queue:
            leaf = min(queue, key=lambda n: (n.last_access, n.serial))
            queue.remove(leaf)
            if leaf.ref_count > 0:
                continue
            for p in leaf.block_ids:
                self.pool.block_release(p)
            released += len(leaf.block_ids)
            parent = leaf.parent
            del parent.children[tuple(leaf.prefix_tokens[:self.B])]
            # 4: cascading eligibility
            if parent is not self.root and not parent.children and parent.ref_count == 0:
                queue.append(parent)
        return released

    def hit_rate(self) -> float:
        return self.matched_tokens / self.prompt_tokens if self.prompt_tokens else 0.0

    def export(self):
        """Preorder, children by ascending first-block tokens: list of
        (parent row, blocks, ref_count, last_access, serial, tokens, block_ids)."""
        rows = []

        def visit(node, parent_row):
            for key in sorted(node.children):
                c = node.children[key]
                row = len(rows)
                rows.append((parent_row, len(c.block_ids), c.ref_count, c.last_access, c.serial,
                             list(c.prefix_tokens), list(c.block_ids)))
                visit(c, row)

        visit(self.root, -1)
        return rows

    def destroy(self) -> None:
        for n in list(self._preorder()):
            for p in n.block_ids:
                self.pool.block_release(p)
        self.root.children = {}

    def _preorder(self):
        out = []

        def visit(node):
            for key in sorted(node.children):
                out.append(node.children[key])
                visit(node.children[key])

        visit(self.root)
        return out
