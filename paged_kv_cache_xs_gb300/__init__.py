"""GB300-native paged-KV decode step: KV append + paged decode attention."""
