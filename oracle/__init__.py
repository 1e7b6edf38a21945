"""Float64 CPU oracle for the MLA paged decode path.

TEST INFRASTRUCTURE ONLY.  It is imported, called or executed by the tests,
``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` / reference arm,
and by nothing else.  The CUDA path never touches it, and it shares no code,
headers, tables or helpers with that path.

Modules:
  formats      -- bf16 / fp8 e4m3fn decoders from the bit definitions
  mla_oracle   -- the attention definition (mla_decode) and the LSE merge
  plan_oracle  -- the work/split plan specification, in plain Python integers
  cache_write  -- the KV-cache write (bf16 / saturating fp8 rows into pool slots)
  rope_cache   -- fused decode RoPE + q concat + cache write
  absorb_bmm   -- the per-head absorb / un-absorb products either side of the decode
"""
