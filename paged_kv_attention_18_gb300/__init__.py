"""GB300 (sm_103a) paged KV attention step: KV scatter + paged attention, via a C ABI."""
