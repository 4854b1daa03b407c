"""Oracle of the adaptive expert cache's planner and of the STRP profile format.

TEST INFRASTRUCTURE ONLY: tests/ may import this module; the library package
must not. Plain Python, one step at a time, in the order the page gives them
("extended-strata-moe reference", section "The adaptive cache", and section
"Profile format (STRP)"); it shares no code with the library's planner.

The rules it restates:
  * heat per (layer, expert): a window adds one pick to each distinct expert
    it routes to, unless it has more rows than the window limit (a large
    batch does not count); heat fades by half every half_life generated
    tokens;
  * every fill period, free slots take the hottest experts not held (up to a
    cap); every round period, the hottest experts not held replace the coldest
    held ones (up to a cap), an incoming expert needing more than ratio times
    the evicted expert's heat plus a number of picks;
  * layers holding every expert are left alone.
Readings taken where the page is silent (the same as the library's, stated in
the design notes): ties go to the lower layer, then the lower expert id; a
swap round skips layers that still have free slots; one advance runs each due
round once, the fill round first; the hysteresis test is computed as
(heat_in - picks) > ratio * heat_out.
"""
from __future__ import annotations

import math
import struct


class CacheOracle:
    def __init__(self, n_layers, n_experts, slots, half_life_tokens=350.0, round_every_tokens=32,
                 max_swaps=64, fill_every_tokens=8, max_fills=128, in_ratio=1.5, in_picks=2.0,
                 max_window_tokens=32):
        self.L, self.E = n_layers, n_experts
        self.slots = [int(s) for s in slots]
        self.half_life = float(half_life_tokens)
        self.round_every, self.max_swaps = round_every_tokens, max_swaps
        self.fill_every, self.max_fills = fill_every_tokens, max_fills
        self.ratio, self.picks = float(in_ratio), float(in_picks)
        self.max_window = max_window_tokens
        self.heat = [[0.0] * n_experts for _ in range(n_layers)]
        # owner[l][s] = expert in slot s of layer l, or -1
        self.owner = [[-1] * self.slots[l] for l in range(n_layers)]
        self.clock = 0
        self.next_fill = fill_every_tokens
        self.next_round = round_every_tokens
        self.swapped = 0

    # ------------------------------------------------------------- queries
    def slot_of(self, l, e):
        for s, x in enumerate(self.owner[l]):
            if x == e:
                return s
        return -1

    def slot_map(self, l):
        return [self.slot_of(l, e) for e in range(self.E)]

    def held(self, l):
        return [x for x in self.owner[l] if x >= 0]

    def is_whole(self, l):
        return len(self.held(l)) >= self.E

    # ------------------------------------------------------------- inputs
    def set_resident(self, l, experts):
        self.owner[l] = [-1] * self.slots[l]
        for s, e in enumerate(experts):
            self.owner[l][s] = int(e)

    def observe(self, l, ids_rows):
        """ids_rows: the window's rows, each a list of k expert ids."""
        if len(ids_rows) > self.max_window:
            return
        picked = set()
        for row in ids_rows:
            for e in row:
                picked.add(int(e))
        for e in picked:
            self.heat[l][e] = self.heat[l][e] + 1.0

    def observe_counts(self, counts):
        """counts[l][e]: picks counted outside the planner (one per expert and
        window), added to the heats as they stand."""
        for l in range(len(self.heat)):
            for e in range(self.E):
                c = int(counts[l][e])
                assert c >= 0
                self.heat[l][e] = self.heat[l][e] + float(c)

    def _cold_hot_lists(self, l):
        """(not held with heat > 0, hottest first), (held, coldest first); ties: lower id."""
        held = set(self.held(l))
        h = self.heat[l]
        outside = [e for e in range(self.E) if e not in held and h[e] > 0.0]
        outside.sort(key=lambda e: (-h[e], e))
        inside = sorted(held, key=lambda e: (h[e], e))
        return outside, inside

    def _fill(self):
        moves = []
        for l in range(self.L):
            if self.is_whole(l):
                continue
            free = [s for s in range(self.slots[l]) if self.owner[l][s] < 0]
            outside, _ = self._cold_hot_lists(l)
            for i in range(min(len(free), len(outside))):
                moves.append((self.heat[l][outside[i]], l, outside[i], -1, free[i]))
        moves.sort(key=lambda m: (-m[0], m[1], m[2]))
        moves = moves[:self.max_fills]
        out = []
        for _, l, e_in, e_out, s in moves:
            self.owner[l][s] = e_in
            out.append((l, s, e_in, -1))
        self.swapped += len(out)
        return out

    def _swap(self, cap):
        moves = []
        for l in range(self.L):
            if self.slots[l] == 0 or self.is_whole(l) or len(self.held(l)) < self.slots[l]:
                continue
            outside, inside = self._cold_hot_lists(l)
            for i in range(min(len(outside), len(inside))):
                h_in, h_out = self.heat[l][outside[i]], self.heat[l][inside[i]]
                if not ((h_in - self.picks) > self.ratio * h_out):
                    break
                moves.append((h_in, l, outside[i], inside[i], self.slot_of(l, inside[i])))
        moves.sort(key=lambda m: (-m[0], m[1], m[2]))
        moves = moves[:cap]
        out = []
        for _, l, e_in, e_out, s in moves:
            self.owner[l][s] = e_in
            out.append((l, s, e_in, e_out))
        self.swapped += len(out)
        return out

    def advance(self, n_tokens):
        if n_tokens > 0:
            f = math.pow(2.0, -float(n_tokens) / self.half_life)
            for l in range(self.L):
                for e in range(self.E):
                    self.heat[l][e] = self.heat[l][e] * f
        self.clock += n_tokens
        out = []
        if self.clock >= self.next_fill:
            out += self._fill()
            self.next_fill = (self.clock // self.fill_every + 1) * self.fill_every
        if self.clock >= self.next_round:
            out += self._swap(self.max_swaps)
            self.next_round = (self.clock // self.round_every + 1) * self.round_every
        return out

    def rebalance(self, max_swaps):
        return self._swap(max_swaps)

    # ------------------------------------------------------------- STRP
    def profile_bytes(self):
        pairs = [(self.heat[l][e], l, e) for l in range(self.L) for e in range(self.E)
                 if self.heat[l][e] > 0.0]
        pairs.sort(key=lambda t: (-t[0], t[1], t[2]))
        rank = [[-1] * self.E for _ in range(self.L)]
        for i, (_, l, e) in enumerate(pairs):
            rank[l][e] = i
        b = b"STRP" + struct.pack("<5I", 1, self.L, self.E, sum(self.slots), len(pairs))
        for _, l, e in pairs:
            b += struct.pack("<2H", l, e)
        for l in range(self.L):
            for e in range(self.E):
                b += struct.pack("<i", rank[l][e])
        return b

    def load_profile(self, data):
        """Raises ValueError for a profile the page's validation rejects."""
        if len(data) < 24 or data[:4] != b"STRP":
            raise ValueError("bad magic")
        version, L, E, _slots, n_ranked = struct.unpack_from("<5I", data, 4)
        if version != 1:
            raise ValueError("bad version")
        if L != self.L or E != self.E:
            raise ValueError("dimensions differ from the model")
        if n_ranked > L * E or len(data) < 24 + 4 * n_ranked:
            raise ValueError("bad pair count")
        pairs = [struct.unpack_from("<2H", data, 24 + 4 * i) for i in range(n_ranked)]
        for l, e in pairs:
            if l >= L or e >= E:
                raise ValueError("pair out of range")
        self.owner = [[-1] * self.slots[l] for l in range(self.L)]
        for l, e in pairs:
            if e in self.owner[l] or -1 not in self.owner[l]:
                continue
            self.owner[l][self.owner[l].index(-1)] = e
