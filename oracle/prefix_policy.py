"""Plain model of the prefix-state cache with second-hit admission.

TEST INFRASTRUCTURE.  Only ``tests/`` may import this module; the library
never does, and this module imports nothing of the library.

Source: "vLLM Kimi K3 지원" (agentlenshq.com), section "하이브리드 KV-Cache
관리" (the recurrent-state blocks are kept apart from prefix matching, so a
prompt that shares a prefix reuses the KDA state saved at that prefix) and
section "에이전틱 캐시 유지 정책" (Marconi-style selective retention: the KDA
state of a prefix is saved only when that prefix is hit for the second time,
so only prefixes that recur take cache room).

The page states the rule, not its mechanics.  Readings taken here (the
plainest ones that fit a chunked prefill whose checkpoints sit on chunk ends):

1. A prefix is the first i * block tokens of a prompt (block a multiple of the
   chunk length); only such prefixes are tracked, so a saved state is always a
   checkpoint at a chunk end and resuming from it keeps the chunk grid.
2. Every plan counts one hit on each block prefix of its prompt, including
   the prompt's full length when that is a whole number of blocks.
3. Reuse: the longest saved prefix of the prompt that still leaves at least
   one token to compute (length <= n - 1).
4. Admission: after counting, the longest prefix of the prompt that is longer
   than the reused one, has at least two hits and holds no state is saved
   during this prompt's prefill, at most one per plan.
5. Slots for saved states come from the cache's own list, lowest first; with
   none free the least recently used saved prefix gives its slot up (never
   the one this plan reuses) and is tracked again as unsaved with its hit
   count; with no such victim nothing is admitted.
6. "Recently used" is one counter stamped on a prefix each time a plan counts
   it, prefixes in increasing length; unsaved prefixes beyond ``max_tracked``
   are dropped least recent first, after the admission.
"""

from __future__ import annotations


class PrefixPolicy:
    def __init__(self, block: int, slots, max_tracked: int):
        if block <= 0 or block % 64 != 0:
            raise ValueError("block must be a positive multiple of 64")
        self.block = block
        self.free = sorted(int(s) for s in slots)
        self.max_tracked = int(max_tracked)
        self.entries = {}  # prefix tuple -> [hits, slot (-1: unsaved), stamp]
        self.clock = 0

    def plan(self, tokens):
        """(hit_len, hit_slot, admit_pos, admit_slot); -1 where there is none."""
        tokens = tuple(int(t) for t in tokens)
        n, B = len(tokens), self.block
        nb = n // B
        # 3. reuse: longest saved prefix of at most n - 1 tokens
        hit = 0
        for i in range((n - 1) // B if n > 0 else 0, 0, -1):
            e = self.entries.get(tokens[:i * B])
            if e is not None and e[1] >= 0:
                hit = i
                break
        # 2 and 6. count a hit on every block prefix, shortest first
        for i in range(1, nb + 1):
            e = self.entries.setdefault(tokens[:i * B], [0, -1, 0])
            e[0] += 1
            self.clock += 1
            e[2] = self.clock
        # 4. admission
        admit, slot = 0, -1
        for i in range(nb, hit, -1):
            e = self.entries[tokens[:i * B]]
            if e[0] >= 2 and e[1] < 0:
                admit = i
                break
        if admit:
            if self.free:
                slot = self.free.pop(0)
            else:
                keep = tokens[:hit * B] if hit else None
                saved = [(e[2], p) for p, e in self.entries.items() if e[1] >= 0 and p != keep]
                if saved:
                    _, victim = min(saved)
                    slot = self.entries[victim][1]
                    self.entries[victim][1] = -1
            if slot >= 0:
                self.entries[tokens[:admit * B]][1] = slot
            else:
                admit = 0
        # 6. bound the unsaved prefixes
        unsaved = sorted((e[2], p) for p, e in self.entries.items() if e[1] < 0)
        for _, p in unsaved[:max(0, len(unsaved) - self.max_tracked)]:
            del self.entries[p]
        hit_slot = self.entries[tokens[:hit * B]][1] if hit else -1
        return (hit * B, hit_slot, admit * B if admit else -1, slot if admit else -1)

    def forget(self, slot: int) -> bool:
        """Gives up the saved state in `slot` (its prefix stays tracked, unsaved)."""
        for e in self.entries.values():
            if e[1] == slot:
                e[1] = -1
                self.free = sorted(self.free + [slot])
                return True
        return False

    def saved(self):
        """{slot: prefix length} of the saved prefixes (for checks)."""
        return {e[1]: len(p) for p, e in self.entries.items() if e[1] >= 0}

    def n_unsaved(self) -> int:
        return sum(1 for e in self.entries.values() if e[1] < 0)
