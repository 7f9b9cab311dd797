"""Oracle restatement of the shard map (step A1).  TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
this module; the product path never imports it.

What it restates, in the pages' order and notation:

* Buffers per (param_dtype, grad_dtype): the Megatron distributed-package page
  (2kiu.com, "Megatron-LM distributed package"), section 2.2 (3): parameters
  are grouped into one _ParamAndGradBuffer per (param dtype, grad dtype), the
  grad dtype being fp32 when grad_reduce_in_fp32 is set.
* Bucketing: the distrib_optimizer page (xiaolong-dev), section "Bucket
  partition: reverse walk + size trigger" and "Two levels of padding": params
  are walked in reverse order; each param start is padded to a multiple of
  64 elements; a param that requires a new bucket first seals the open one;
  a bucket is sealed once param_end - bucket_start >= bucket_size; the tail
  forms the last bucket.  A sealed bucket's end is padded to a multiple of
  lcm(DP, 128), or lcm(DP, 128, 2^16) with pad_buckets_for_high_nccl_busbw.
  The bodies of _pad and _update_bucket_metadata are not printed; the plain
  readings are ceil(x/d)*d and "pad the end, record (offset, padded numel,
  unpadded numel), open the next bucket at the padded end".
* Final size checks: same page, "Final memory size assertions".
* Equal split of a bucket and the four views of each param: same page,
  "Bucket-level equal split" (_build_model_gbuf_range) and "Range class: four
  views" (_build_model_gbuf_param_range_map).
* The worked example of the same page (DP=4, one bucket of 1024 bf16 elements,
  256 elements per rank) is one of the pins of this module.

The flat per-rank shard offset (shard_offset) is the layout convention of the
library's ABI: a rank's shard of a buffer is the concatenation, in bucket
order, of its slice of every bucket.
"""

import math

F32, BF16, F16 = 0, 1, 2


class Range:
    """A half-open index interval [start, end) with a size, shifted by normalize()."""

    __slots__ = ("start", "end")

    def __init__(self, start, end):
        self.start = start
        self.end = end

    @property
    def size(self):
        return self.end - self.start

    def normalize(self, start=0):
        return Range(start, start + self.size)

    def as_tuple(self):
        return (self.start, self.end)

    def __eq__(self, other):
        return isinstance(other, Range) and self.as_tuple() == other.as_tuple()

    def __repr__(self):
        return f"Range({self.start},{self.end})"


def pad_up(x, d):
    """The smallest multiple of d that is >= x."""
    return -(-x // d) * d


class Bucket:
    __slots__ = ("offset", "numel", "numel_unpadded", "params")

    def __init__(self, offset, numel, numel_unpadded, params):
        self.offset = offset
        self.numel = numel
        self.numel_unpadded = numel_unpadded
        self.params = params


class Buffer:
    """One contiguous param-and-grad buffer and its buckets."""

    def __init__(self, param_dtype, grad_dtype, params):
        self.param_dtype = param_dtype
        self.grad_dtype = grad_dtype
        self.params = params  # global param ids, model order
        self.index = {}  # param id -> (start, end, bucket id)
        self.buckets = []
        self.numel = 0
        self.numel_unpadded = 0


def _lay_out(buf, numel, new_bucket, dp, bucket_size, busbw):
    divisor = math.lcm(dp, 128, 2**16) if busbw else math.lcm(dp, 128)
    state = {"open_start": 0, "members": []}

    def seal(end):
        # Close the open bucket at `end` (unpadded) and return its padded end.
        padded = pad_up(end, divisor)
        start = state["open_start"]
        buf.buckets.append(Bucket(start, padded - start, end - start, state["members"]))
        state["open_start"] = padded
        state["members"] = []
        return padded

    cursor = 0
    last_end = 0
    for pid in reversed(buf.params):
        start = pad_up(cursor, 64)
        if new_bucket[pid] and state["members"]:
            start = seal(start)
        end = start + numel[pid]
        buf.index[pid] = (start, end, len(buf.buckets))
        state["members"].append(pid)
        size_trigger = bucket_size is not None and end - state["open_start"] >= bucket_size
        if size_trigger or new_bucket[pid]:
            cursor = seal(end)
        else:
            cursor = end
        last_end = end
    if state["members"]:
        seal(last_end)
    buf.numel = buf.buckets[-1].offset + buf.buckets[-1].numel if buf.buckets else 0
    buf.numel_unpadded = sum(b.numel_unpadded for b in buf.buckets)
    assert buf.numel_unpadded <= buf.numel
    assert buf.numel % dp == 0


class ShardMap:
    """Buffers, buckets and per-rank views of a list of params."""

    def __init__(self, params, dp, bucket_size=None, grad_reduce_in_fp32=False,
                 pad_for_high_busbw=False):
        """params: list of dicts with keys numel, dtype, and optional
        new_bucket (bool) and wd_mult (float).  bucket_size None = no size
        trigger (one bucket unless a param asks for a new one)."""
        assert dp >= 1
        self.dp = dp
        self.params = params
        numel = [p["numel"] for p in params]
        new_bucket = [bool(p.get("new_bucket", False)) for p in params]
        groups = {}
        for pid, p in enumerate(params):
            gdt = F32 if grad_reduce_in_fp32 else p["dtype"]
            groups.setdefault((p["dtype"], gdt), []).append(pid)
        self.buffers = []
        for (pdt, gdt), pids in groups.items():
            buf = Buffer(pdt, gdt, pids)
            _lay_out(buf, numel, new_bucket, dp, bucket_size, pad_for_high_busbw)
            self.buffers.append(buf)

    def bucket_world_range(self, bi, b, r):
        """Rank r's slice of bucket b of buffer bi, in buffer coordinates."""
        bucket = self.buffers[bi].buckets[b]
        s = bucket.numel // self.dp
        lo = r * s
        hi = min(bucket.numel, lo + s)
        return Range(lo + bucket.offset, hi + bucket.offset)

    def shard_numel(self, bi):
        return self.buffers[bi].numel // self.dp

    def bucket_shard_base(self, bi, b):
        """Offset of bucket b's slice inside a rank's flat shard of buffer bi."""
        return sum(bk.numel // self.dp for bk in self.buffers[bi].buckets[:b])

    def rank_views(self, bi, b, r):
        """The four views of every param that meets rank r's slice of bucket b.

        Returns {param id: {"gbuf_world", "gbuf_world_in_bucket", "gbuf_local",
        "param": Range, "shard_offset": int}}."""
        buf = self.buffers[bi]
        bucket = buf.buckets[b]
        world = self.bucket_world_range(bi, b, r)
        base = self.bucket_shard_base(bi, b)
        views = {}
        for pid, (p_start, p_end, _) in buf.index.items():
            lo = max(0, p_start - world.start)
            hi = min(world.size, p_end - world.start)
            if hi <= lo:
                continue
            local = Range(lo, hi)
            in_world = local.normalize(lo + world.start)
            views[pid] = {
                "gbuf_world": in_world,
                "gbuf_world_in_bucket": Range(in_world.start - bucket.offset,
                                              in_world.end - bucket.offset),
                "gbuf_local": local,
                "param": local.normalize(max(0, world.start - p_start)),
                "shard_offset": base + local.start,
            }
        return views

    def rank_pieces(self, bi, r):
        """All param pieces of rank r in buffer bi, in shard order:
        list of (param id, bucket id, views)."""
        out = []
        for b in range(len(self.buffers[bi].buckets)):
            vs = self.rank_views(bi, b, r)
            for pid in sorted(vs, key=lambda q: vs[q]["gbuf_local"].start):
                out.append((pid, b, vs[pid]))
        return out
