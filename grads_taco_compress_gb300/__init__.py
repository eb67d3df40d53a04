"""GB300-native TACO fused compress / decompress-reduce operator."""
